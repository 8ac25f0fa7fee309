// decode_simt.cu — split-K decode attention on CUDA cores for the code widths
// packed as a plain bit stream (b in {1, 3, 5, 6, 7}; tract #2329 makes the
// width configurable, the kvquant++ README recommends 3 bits).
//
// The tensor-core kernel (decode_mma.cuh) turns codes into MMA operands with
// one AND per code pair, which needs the word-rule packing of b in {2, 4, 8}
// (both codes of a pair at the same bit of the two halves of a word).  A bit
// stream puts codes at arbitrary bit offsets, so this kernel dequantizes on
// CUDA cores instead, in fp32:
//   s_t = Σ_c (q_c Δ_c) code_tc + Σ_c q_c min_c      (keys, per channel)
//   o_c = Σ_t (p_t Δ_t) code_ct + Σ_t p_t min_t      (values, per token)
// with the same online softmax (log2 units) and split-K merge as the
// tensor-core kernel (KV-cache quantization guide (pigeon), "How it works",
// step 5).
//
// Work split: one CTA per (sequence, kv head, split); a unit's items are its
// visible frozen groups, then its tail in chunks of 32 tokens (sinks, ring),
// cut into `splits` contiguous ranges; the CTA's 4 warps take items in turn.
// Per frozen group a warp copies the block to its shared memory, then
//   scores: lane = token, a code row read from shared memory, q_c Δ_c of
//           every head broadcast from shared memory;
//   values: lane = channel (lane + 32 j), p_t Δ_t broadcast.
// All query heads of the kv head share each block read.  The warps' (m, l, o)
// are combined in shared memory; a unit split over several CTAs leaves
// partial records and the last CTA (an atomic count) merges them.
#include "kivi_internal.cuh"

#include <math.h>

namespace kivi {
namespace simt {

constexpr int kWarps = 4;
constexpr int kMaxRep = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTail = 32;   // tail tokens per item

struct Args {
  Geo g;
  const uint8_t* arena;
  const __half* q;
  __half* out;
  float* partials;      // [B * h_q][stride][d + 4]: o[d], m, l, 2 pad
  unsigned* counters;   // [B * h_kv]: CTAs finished per unit
  DecodePlan plan;
  int32_t stride;
  int32_t splits;       // CTAs per unit
  int32_t items;        // items per unit: visible groups + tail chunks
  int32_t sink_items;   // tail chunks of sinks
};

// Shared memory of one warp (floats unless noted): the block bytes, q of
// every head (for tails), q Δ of every head (per group), p Δ (values).
template <int D>
struct Smem {
  __host__ __device__ static int block_bytes(const Geo& g) { return static_cast<int>((g.block_bytes + 15) / 16 * 16); }
  __host__ __device__ static int bytes(const Geo& g) {
    return block_bytes(g) + 4 * (2 * kMaxRep * D + kMaxRep * 64);
  }
};

// Code j of a bit-stream row at `row` (bytes in shared memory, 4-byte aligned
// start is not needed: the read is two aligned 32-bit words around it).
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint8_t* row, int j) {
  const int bit = BITS * j;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(row + (bit >> 3)) & ~uintptr_t(3));
  const int sh = static_cast<int>((reinterpret_cast<uintptr_t>(row + (bit >> 3)) & 3) * 8) + (bit & 7);
  const uint32_t lo = w[0];
  const uint32_t hi = (sh + BITS > 32) ? w[1] : 0u;
  return __funnelshift_r(lo, hi, sh) & ((1u << BITS) - 1u);
}

template <int D, int BITS>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(const Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const Geo& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rep = g.rep;
  const int unit = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int bb = unit / g.hkv, hk = unit % g.hkv;
  const uint8_t* ubase = a.arena + static_cast<int64_t>(unit) * g.unit_bytes;
  const int G = g.G;
  const float qscale = kLog2e * rsqrtf(static_cast<float>(D));
  constexpr int CPL = D / 32;   // channels per lane (values)

  uint8_t* my = smem + warp * Smem<D>::bytes(g);
  uint8_t* blk = my;
  float* qs = reinterpret_cast<float*>(my + Smem<D>::block_bytes(g));   // [rep][D] q * qscale
  float* qd = qs + kMaxRep * D;                                        // [rep][D] q Δ * qscale
  float* pv = qd + kMaxRep * D;                                        // [rep][64] p Δ or p

  // q of the unit's heads, scaled to log2 units
  for (int i = lane; i < rep * D; i += 32) {
    const int h = i / D, c = i % D;
    qs[i] = __half2float(a.q[(static_cast<int64_t>(bb) * g.hq + hk * rep + h) * D + c]) * qscale;
  }
  __syncwarp();

  float m[kMaxRep], l[kMaxRep], o[kMaxRep][CPL];
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) o[h][j] = 0.f;
  }
  const int64_t lo_pos = g.window > 0 ? a.plan.q_pos0 + 1 - g.window : INT64_MIN;
  const int n_vis = static_cast<int>(a.plan.n_vis_groups);
  const int i0 = static_cast<int>((static_cast<int64_t>(split) * a.items) / a.splits);
  const int i1 = static_cast<int>((static_cast<int64_t>(split + 1) * a.items) / a.splits);
  const int rs0 = static_cast<int>((a.plan.st.n_groups * g.G) % g.R);
  const int64_t ring_pos0 = g.S + a.plan.st.n_groups * g.G;
  const int n_sink = static_cast<int>(a.plan.st.n_sink), n_res = static_cast<int>(a.plan.st.n_res);

  // online softmax step for head h over this lane's scores s[0..ns) (tokens
  // lane + 32 i), -inf for absent tokens; returns the weights in p
  auto softmax = [&](int h, const float* s, float* p, int ns) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (i < ns) mx = fmaxf(mx, s[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float mn = fmaxf(m[h], mx);
    const float corr = (m[h] == -INFINITY) ? 0.f : exp2f(m[h] - mn);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (i < ns) {
        p[i] = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - mn);
        sum += p[i];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (mn == -INFINITY) return;   // nothing visible yet: every p is 0
    m[h] = mn;
    l[h] = l[h] * corr + sum;
#pragma unroll
    for (int j = 0; j < CPL; ++j) o[h][j] *= corr;
  };

  for (int it = i0 + warp; it < i1; it += kWarps) {
    if (it < n_vis) {
      // ------------------------------------------------ a frozen group
      const int64_t grp = a.plan.g_first + it;
      const int64_t slot = g.window > 0 ? grp % g.n_slots : grp;
      const uint4* src = reinterpret_cast<const uint4*>(ubase + g.groups + slot * g.block_bytes);
      for (int i = lane; i < static_cast<int>(g.block_bytes / 16); i += 32)
        reinterpret_cast<uint4*>(blk)[i] = src[i];
      __syncwarp();
      const __half* ks = reinterpret_cast<const __half*>(blk + g.blk_ks);   // Δ[D], min[D]
      const __half* vs = reinterpret_cast<const __half*>(blk + g.blk_vs);   // (Δ, min) per token
      // q Δ per head and channel; Σ q min per head
      float cmin[kMaxRep];
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) cmin[h] = 0.f;
      for (int c = lane; c < D; c += 32) {
        const float dq = __half2float(ks[c]), mn = __half2float(ks[D + c]);
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          if (h < rep) {
            qd[h * D + c] = qs[h * D + c] * dq;
            cmin[h] = fmaf(qs[h * D + c], mn, cmin[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cmin[h] += __shfl_xor_sync(0xffffffffu, cmin[h], off);
      __syncwarp();
      const int64_t a0 = g.S + grp * G;
      // scores: lane = token t = lane + 32 i (heads unrolled so that the
      // per-head state stays in registers)
      constexpr int kMaxTl = 2;   // G <= 64
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        if (h >= rep) break;
        float s[kMaxTl], p[kMaxTl] = {0.f, 0.f};
        const int ns = (G + 31) / 32;
#pragma unroll
        for (int i = 0; i < kMaxTl; ++i) {
          if (i >= ns) break;
          const int t = lane + 32 * i;
          s[i] = -INFINITY;
          if (t < G && a0 + t >= lo_pos) {
            const uint8_t* row = blk + g.blk_kq + t * (D * BITS / 8);
            const float* qh = qd + h * D;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc = fmaf(qh[c], static_cast<float>(code_at<BITS>(row, c)), acc);
            s[i] = acc + cmin[h];
          }
        }
        softmax(h, s, p, ns);
        // p Δ_t into shared memory, Σ p min_t per lane's tokens
        float pmin = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxTl; ++i) {
          if (i >= ns) break;
          const int t = lane + 32 * i;
          if (t < G) {
            const float vd = __half2float(vs[2 * t]), vm = __half2float(vs[2 * t + 1]);
            pv[h * 64 + t] = p[i] * vd;
            pmin = fmaf(p[i], vm, pmin);
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) pmin += __shfl_xor_sync(0xffffffffu, pmin, off);
        __syncwarp();
        // values: lane = channel lane + 32 j
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const int c = lane + 32 * j;
          const uint8_t* row = blk + g.blk_vq + c * (G * BITS / 8);
          float acc = pmin;
          for (int t = 0; t < G; ++t) acc = fmaf(pv[h * 64 + t], static_cast<float>(code_at<BITS>(row, t)), acc);
          o[h][j] += acc;
        }
        __syncwarp();
      }
    } else {
      // ------------------------------------------------ a tail chunk of up to 32 tokens
      const int tc = it - n_vis;
      const bool sink = tc < a.sink_items;
      const int first = sink ? kTail * tc : kTail * (tc - a.sink_items);
      const int n = sink ? min(kTail, n_sink - first) : min(kTail, n_res - first);
      if (n <= 0) continue;
      const int t = lane;   // token first + t
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        if (h >= rep) break;
        float s[1], p[1];
        s[0] = -INFINITY;
        if (t < n) {
          float acc = 0.f;
          const float* qh = qs + h * D;
          if (sink) {
            const float* kr = reinterpret_cast<const float*>(ubase + g.sink_k) + static_cast<int64_t>(first + t) * D;
            for (int c = 0; c < D; ++c) acc = fmaf(qh[c], kr[c], acc);
          } else {
            const int slot = (rs0 + first + t) % g.R;
            const __half* kr = reinterpret_cast<const __half*>(ubase + g.res_k) + static_cast<int64_t>(slot) * D;
            for (int c = 0; c < D; ++c) acc = fmaf(qh[c], __half2float(kr[c]), acc);
          }
          const int64_t pos = sink ? first + t : ring_pos0 + first + t;
          (void)pos;   // every sink and ring token lies inside any window (W >= R)
          s[0] = acc;
        }
        softmax(h, s, p, 1);
        pv[h * 64 + lane] = (t < n) ? p[0] : 0.f;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const int c = lane + 32 * j;
          float acc = 0.f;
          for (int u = 0; u < n; ++u) {
            float v;
            if (sink) {
              v = reinterpret_cast<const float*>(ubase + g.sink_v)[static_cast<int64_t>(first + u) * D + c];
            } else {
              const int slot = (rs0 + first + u) % g.R;
              v = __half2float(reinterpret_cast<const __half*>(ubase + g.res_v)[static_cast<int64_t>(slot) * D + c]);
            }
            acc = fmaf(pv[h * 64 + u], v, acc);
          }
          o[h][j] += acc;
        }
        __syncwarp();
      }
    }
  }

  // ---------------------------------------------------- combine the warps
  __syncthreads();   // block buffers are free now: reuse the CTA's shared memory
  float* cm = reinterpret_cast<float*>(smem);                      // [warps][rep] m
  float* cl = cm + kWarps * kMaxRep;                               // [warps][rep] l
  float* co = cl + kWarps * kMaxRep;                               // [warps][rep][D] o
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    if (h >= rep) break;
    if (lane == 0) { cm[warp * kMaxRep + h] = m[h]; cl[warp * kMaxRep + h] = l[h]; }
#pragma unroll
    for (int j = 0; j < CPL; ++j) co[(warp * kMaxRep + h) * D + lane + 32 * j] = o[h][j];
  }
  __syncthreads();
  __shared__ unsigned s_last;
  const bool single = a.splits == 1;
  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * kMaxRep + h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        const float mw = cm[w * kMaxRep + h];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        L = fmaf(cl[w * kMaxRep + h], f, L);
        O = fmaf(co[(w * kMaxRep + h) * D + c], f, O);
      }
    }
    const int64_t row = static_cast<int64_t>(bb) * g.hq + hk * rep + h;
    if (single) {
      a.out[row * D + c] = __float2half_rn(L > 0.f ? O / L : 0.f);
    } else {
      float* dst = a.partials + (row * a.stride + split) * (D + 4);
      dst[c] = O;
      if (c == 0) { dst[D] = M; dst[D + 1] = L; }
    }
  }
  if (single) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counters + unit, 1u) == static_cast<unsigned>(a.splits - 1)) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const int64_t row = static_cast<int64_t>(bb) * g.hq + hk * rep + h;
    const float* base = a.partials + row * a.stride * (D + 4);
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, __ldcg(base + s * (D + 4) + D));
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.splits; ++s) {
        const float ms = __ldcg(base + s * (D + 4) + D);
        const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
        L = fmaf(__ldcg(base + s * (D + 4) + D + 1), f, L);
        O = fmaf(__ldcg(base + s * (D + 4) + c), f, O);
      }
    }
    a.out[row * D + c] = __float2half_rn(L > 0.f ? O / L : 0.f);
  }
  if (threadIdx.x == 0) a.counters[unit] = 0u;
}

template <int D, int BITS>
cudaError_t launch_one(const Args& a, int ctas, int smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<D, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_simt_kernel<D, BITS><<<ctas, kWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Args& a, int ctas, int smem, cudaStream_t s) {
  switch (a.g.bits) {
    case 1: return launch_one<D, 1>(a, ctas, smem, s);
    case 3: return launch_one<D, 3>(a, ctas, smem, s);
    case 5: return launch_one<D, 5>(a, ctas, smem, s);
    case 6: return launch_one<D, 6>(a, ctas, smem, s);
    case 7: return launch_one<D, 7>(a, ctas, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace simt

cudaError_t launch_decode_simt(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                               const DecodePlan& plan, float* partials, int32_t stride, unsigned* counters,
                               int32_t target_ctas, cudaStream_t stream) {
  if (g.G > 64 || g.rep > simt::kMaxRep || stride < 3) return cudaErrorInvalidValue;
  simt::Args a{};
  a.g = g;
  a.arena = arena;
  a.q = q;
  a.out = out;
  a.partials = partials;
  a.counters = counters;
  a.plan = plan;
  a.stride = stride;
  a.sink_items = static_cast<int32_t>((plan.st.n_sink + simt::kTail - 1) / simt::kTail);
  a.items = static_cast<int32_t>(plan.n_vis_groups) + a.sink_items +
            static_cast<int32_t>((plan.st.n_res + simt::kTail - 1) / simt::kTail);
  if (a.items < 1) a.items = 1;
  const int64_t units = static_cast<int64_t>(g.B) * g.hkv;
  int64_t splits = (target_ctas + units - 1) / units;
  if (splits > a.items) splits = a.items;
  if (splits > stride) splits = stride;
  if (splits < 1) splits = 1;
  a.splits = static_cast<int32_t>(splits);
  const int smem = simt::kWarps * (g.d == 64 ? simt::Smem<64>::bytes(g) : simt::Smem<128>::bytes(g));
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  const int ctas = static_cast<int>(units * splits);
  return g.d == 64 ? simt::launch_d<64>(a, ctas, smem, stream) : simt::launch_d<128>(a, ctas, smem, stream);
}

}  // namespace kivi
