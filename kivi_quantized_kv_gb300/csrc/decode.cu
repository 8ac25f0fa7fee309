// decode.cu — split-K decode attention over the packed KIVI cache (sm_103a).
//
// softmax(q Kᵀ / sqrt(d)) V with K and V dequantized group by group on the
// fly, never materialising an fp16 copy (KV-cache quantization guide
// (pigeon), "How it works", step 5); query heads share their kv head (GQA,
// tract #2329 "What's in the PR").
//
// Grid (split, kv head, sequence); 4 warps per CTA.  A split owns a range of
// frozen groups; the last split also owns the sinks and the ring.  Per frozen
// group the key dot product folds the per-channel scale into the query,
//   q·k̂_t = Σ_c (q_c Δ_c) code_tc + Σ_c q_c min_c,
// and the value sum folds the per-token scale into the probability,
//   Σ_t p_t v̂_tc = Σ_t (p_t Δ_t) code_tc + Σ_t p_t min_t,
// both exact rearrangements of the dequantized sums.  Each warp keeps an
// online softmax (running max m, sum l, output o) per query head; the CTA
// combines its warps and writes one partial (o, m, l) per head; merge_kernel
// combines the splits and writes fp16 out.
#include "kivi_internal.cuh"

#include <math.h>

namespace kivi {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxRep = 8;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float code_to_float(uint32_t c) {
  return __uint_as_float(0x4B000000u | c) - 8388608.0f;   // exact for c < 2^23
}

// Element j of a packed row: word j / per, half j & 1, bit b * ((j % per) >> 1).
template <int BITS>
__device__ __forceinline__ uint32_t extract(uint32_t word, int jj) {
  return (word >> (16 * (jj & 1) + BITS * (jj >> 1))) & ((1u << BITS) - 1u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct WarpSmem {
  float qd[128 * kMaxRep];   // q_c Δ_c (log2 e / sqrt(d) folded), [c][h]
  float pd[32 * kMaxRep];    // p_t Δ_t for the current token chunk, [t][h]
};

template <int D, int BITS>
__global__ void __launch_bounds__(kWarps * 32)
decode_v0_kernel(Geo g, const uint8_t* __restrict__ arena, const __half* __restrict__ q,
                 float* __restrict__ part, DecodePlan plan) {
  constexpr int NC = D / 32;            // channels per lane
  constexpr int PER = 32 / BITS;        // codes per 32-bit word
  __shared__ float qs[kMaxRep][D];      // q (log2 e / sqrt(d) folded)
  __shared__ WarpSmem ws[kWarps];
  __shared__ float red_m[kWarps][kMaxRep], red_l[kWarps][kMaxRep];
  __shared__ float red_o[kWarps][kMaxRep][D];

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rep = g.rep;
  const float qscale = kLog2e * rsqrtf(static_cast<float>(D));
  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    qs[r][c] = __half2float(q[(static_cast<int64_t>(b) * g.hq + h * rep + r) * D + c]) * qscale;
  }
  __syncthreads();

  const uint8_t* unit = arena + (static_cast<int64_t>(b) * g.hkv + h) * g.unit_bytes;
  const int64_t T = plan.st.T;
  const int64_t lo = g.window > 0 ? T - g.window : 0;   // window start (sinks always visible)

  float m[kMaxRep], l_lane[kMaxRep], mn_acc[kMaxRep], o[kMaxRep][NC];
#pragma unroll
  for (int r = 0; r < kMaxRep; ++r) {
    m[r] = -INFINITY; l_lane[r] = 0.f; mn_acc[r] = 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) o[r][j] = 0.f;
  }

  // ---- frozen groups ----
  const int64_t ga = plan.g_first + static_cast<int64_t>(split) * plan.groups_per_split;
  int64_t gb = ga + plan.groups_per_split;
  if (gb > plan.g_first + plan.n_vis_groups) gb = plan.g_first + plan.n_vis_groups;
  WarpSmem& sm = ws[warp];
  for (int64_t grp = ga + warp; grp < gb; grp += kWarps) {
    const uint8_t* blk = unit + g.groups + (grp % g.n_slots) * g.block_bytes;
    const __half* kdelta = reinterpret_cast<const __half*>(blk + g.blk_ks);
    const __half* kmin = kdelta + D;
    // per-group folded query q_c Δ_c and the constant Σ_c q_c min_c
    float cst[kMaxRep];
#pragma unroll
    for (int r = 0; r < kMaxRep; ++r) cst[r] = 0.f;
    for (int c = lane; c < D; c += 32) {
      const float dk = __half2float(kdelta[c]), mk = __half2float(kmin[c]);
#pragma unroll
      for (int r = 0; r < kMaxRep; ++r) {
        if (r < rep) {
          sm.qd[c * kMaxRep + r] = qs[r][c] * dk;
          cst[r] = fmaf(qs[r][c], mk, cst[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRep; ++r) cst[r] = warp_sum(cst[r]);
    __syncwarp();
    const int64_t a0 = g.S + grp * g.G;
    for (int t0 = 0; t0 < g.G; t0 += 32) {
      const int t = t0 + lane;
      const bool valid = (t < g.G) && (a0 + t >= lo);
      // scores: lane owns token t
      float s[kMaxRep];
#pragma unroll
      for (int r = 0; r < kMaxRep; ++r) s[r] = cst[r];
      if (t < g.G) {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(blk + g.blk_kq + static_cast<int64_t>(t) * D * BITS / 8);
#pragma unroll 4
        for (int w = 0; w < D / PER; ++w) {
          const uint32_t word = row[w];
#pragma unroll
          for (int jj = 0; jj < PER; ++jj) {
            const float cf = code_to_float(extract<BITS>(word, jj));
            const float* qd = &sm.qd[(w * PER + jj) * kMaxRep];
#pragma unroll
            for (int r = 0; r < kMaxRep; ++r)
              if (r < rep) s[r] = fmaf(qd[r], cf, s[r]);
          }
        }
      }
      // online softmax over the chunk, per head
      const __half* vsc = reinterpret_cast<const __half*>(blk + g.blk_vs);
      const float vd = (t < g.G) ? __half2float(vsc[2 * t]) : 0.f;
      const float vm = (t < g.G) ? __half2float(vsc[2 * t + 1]) : 0.f;
#pragma unroll
      for (int r = 0; r < kMaxRep; ++r) {
        if (r >= rep) continue;
        const float cm = warp_max(valid ? s[r] : -INFINITY);
        const float mnew = fmaxf(m[r], cm);
        const float corr = (m[r] == -INFINITY) ? 0.f : exp2f(m[r] - mnew);
        const float p = valid ? exp2f(s[r] - mnew) : 0.f;
        m[r] = mnew;
        l_lane[r] = l_lane[r] * corr + p;
        mn_acc[r] = mn_acc[r] * corr + p * vm;
#pragma unroll
        for (int j = 0; j < NC; ++j) o[r][j] *= corr;
        sm.pd[lane * kMaxRep + r] = p * vd;
      }
      __syncwarp();
      // values: lane owns channels c = lane + 32 j; row c holds the group's tokens
      const int nt = (g.G - t0) < 32 ? (g.G - t0) : 32;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int c = lane + 32 * j;
        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(blk + g.blk_vq + static_cast<int64_t>(c) * g.G * BITS / 8);
        for (int w = 0; w < nt / PER; ++w) {
          const uint32_t word = vrow[(t0 / PER) + w];
#pragma unroll
          for (int jj = 0; jj < PER; ++jj) {
            const float cf = code_to_float(extract<BITS>(word, jj));
            const float* pd = &sm.pd[(w * PER + jj) * kMaxRep];
#pragma unroll
            for (int r = 0; r < kMaxRep; ++r)
              if (r < rep) o[r][j] = fmaf(pd[r], cf, o[r][j]);
          }
        }
      }
      __syncwarp();
    }
  }

  // ---- sinks and ring (last split): one token at a time, lanes own channels ----
  if (split == plan.splits - 1) {
    const int64_t n_sink = plan.st.n_sink;
    const int64_t r0 = g.S + plan.st.n_groups * g.G;   // first ring token
    const int64_t n_items = n_sink + plan.st.n_res;
    for (int64_t it = warp; it < n_items; it += kWarps) {
      const int64_t a = (it < n_sink) ? it : r0 + (it - n_sink);
      if (a >= g.S && a < lo) continue;
      float kv[NC], vv[NC];
      if (a < g.S) {
        const float* kr = reinterpret_cast<const float*>(unit + g.sink_k) + a * D;
        const float* vr = reinterpret_cast<const float*>(unit + g.sink_v) + a * D;
#pragma unroll
        for (int j = 0; j < NC; ++j) { kv[j] = kr[lane + 32 * j]; vv[j] = vr[lane + 32 * j]; }
      } else {
        const int64_t slot = (a - g.S) % g.R;
        const __half* kr = reinterpret_cast<const __half*>(unit + g.res_k) + slot * D;
        const __half* vr = reinterpret_cast<const __half*>(unit + g.res_v) + slot * D;
#pragma unroll
        for (int j = 0; j < NC; ++j) { kv[j] = __half2float(kr[lane + 32 * j]); vv[j] = __half2float(vr[lane + 32 * j]); }
      }
#pragma unroll
      for (int r = 0; r < kMaxRep; ++r) {
        if (r >= rep) continue;
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j) part = fmaf(qs[r][lane + 32 * j], kv[j], part);
        const float sc = warp_sum(part);
        const float mnew = fmaxf(m[r], sc);
        const float corr = (m[r] == -INFINITY) ? 0.f : exp2f(m[r] - mnew);
        const float p = exp2f(sc - mnew);
        m[r] = mnew;
        l_lane[r] = l_lane[r] * corr + (lane == 0 ? p : 0.f);
        mn_acc[r] *= corr;
#pragma unroll
        for (int j = 0; j < NC; ++j) o[r][j] = fmaf(o[r][j], corr, p * vv[j]);
      }
    }
  }

  // ---- combine warps, write the CTA's partial per head ----
#pragma unroll
  for (int r = 0; r < kMaxRep; ++r) {
    if (r >= rep) continue;
    const float l = warp_sum(l_lane[r]);
    const float mnt = warp_sum(mn_acc[r]);
    if (lane == 0) { red_m[warp][r] = m[r]; red_l[warp][r] = l; }
#pragma unroll
    for (int j = 0; j < NC; ++j) red_o[warp][r][lane + 32 * j] = o[r][j] + mnt;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][r]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        if (red_m[w][r] == -INFINITY) continue;
        const float f = exp2f(red_m[w][r] - M);
        L += red_l[w][r] * f;
        O += red_o[w][r][c] * f;
      }
    }
    float* dst = part + ((static_cast<int64_t>(b) * g.hq + h * rep + r) * g.max_splits + split) * (D + 2);
    dst[c] = O;
    if (c == 0) { dst[D] = M; dst[D + 1] = L; }
  }
}

// Combines the splits of one (sequence, query head): M = max m_i,
// L = Σ l_i 2^(m_i - M), out = Σ o_i 2^(m_i - M) / L (m in log2 units).
template <int D>
__global__ void merge_kernel(Geo g, const float* __restrict__ partials, __half* __restrict__ out, int splits) {
  const int hq = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const float* part = partials + (static_cast<int64_t>(b) * g.hq + hq) * g.max_splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part[s * (D + 2) + D]);
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ms = part[s * (D + 2) + D];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - M);
      L += part[s * (D + 2) + D + 1] * f;
      O += part[s * (D + 2) + c] * f;
    }
  }
  out[(static_cast<int64_t>(b) * g.hq + hq) * D + c] = __float2half_rn(L > 0.f ? O / L : 0.f);
}

template <int D, int BITS>
cudaError_t launch_v0(const Geo& g, const uint8_t* arena, const __half* q, __half* out, const DecodePlan& plan,
                      float* partials, cudaStream_t stream) {
  dim3 grid(plan.splits, g.hkv, g.B);
  decode_v0_kernel<D, BITS><<<grid, kWarps * 32, 0, stream>>>(g, arena, q, partials, plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  merge_kernel<D><<<dim3(g.hq, g.B), D, 0, stream>>>(g, partials, out, plan.splits);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_scratch(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                  const DecodePlan& plan, float* partials, unsigned* counters,
                                  cudaStream_t stream) {
  (void)counters;   // the separate merge pass needs no counters
  if (g.rep > kMaxRep) return cudaErrorInvalidValue;
  if (g.d == 64) {
    if (g.bits == 2) return launch_v0<64, 2>(g, arena, q, out, plan, partials, stream);
    if (g.bits == 4) return launch_v0<64, 4>(g, arena, q, out, plan, partials, stream);
    return launch_v0<64, 8>(g, arena, q, out, plan, partials, stream);
  }
  if (g.bits == 2) return launch_v0<128, 2>(g, arena, q, out, plan, partials, stream);
  if (g.bits == 4) return launch_v0<128, 4>(g, arena, q, out, plan, partials, stream);
  return launch_v0<128, 8>(g, arena, q, out, plan, partials, stream);
}

cudaError_t launch_decode(const Geo& g, uint8_t* arena, const __half* q, __half* out,
                          const DecodePlan& plan, cudaStream_t stream) {
  return launch_decode_scratch(g, arena, q, out, plan, reinterpret_cast<float*>(arena + g.ws_partials),
                               reinterpret_cast<unsigned*>(arena + g.ws_counters), stream);
}

}  // namespace kivi
