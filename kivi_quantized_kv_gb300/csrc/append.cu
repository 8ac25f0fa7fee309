// append.cu — the write side of the KIVI cache on sm_103a.
//
// flush_kernel: one CTA per (new frozen group, kv head, sequence).  It stages
// the group's G fp16 tokens (keys and values) in shared memory, quantizes
//   keys   per channel over the G tokens  (KV-cache quantization guide
//          (pigeon), "How it works", step 1),
//   values per token over the d channels  (same page, step 2),
// with q = round((x - min) / Δ), Δ = (max - min) / (2^b - 1) (step 3), and
// writes the packed codes and fp16 (Δ, min) pairs of the group block.  Once a
// block is written it never changes (tract #2458: frozen block scales).
//
// Bit-exactness: every fp32 operation of the quantizer is an explicit
// round-to-nearest-even intrinsic (__fsub_rn, __fdiv_rn, __fadd_rn), so the
// compiler cannot contract or reorder it; fp16 conversion is
// __float2half_rn; "round" is rintf (half to even).  min and max are
// canonicalised with + 0.0f so -0 and +0 give the same bytes.  A code is
// rintf of the correctly rounded quotient (x - min) / Δ, computed through
// the correctly rounded 1/Δ (code_of), which rounds to the same integer.
//
// Dense-and-sparse outliers (when the cache keeps them; pigeon guide, "KVQuant
// adds"): before the quantizer, the n_out values of largest magnitude of the
// key block and of the value block are found by n_out rounds of a block-wide
// maximum over a unique 32-bit key per element, (|x| bits << 16) | (0xFFFF -
// flat index), each round taking the largest key below the previous round's
// (so ties go to the smaller flat index).  They are flagged in a bitmask,
// left out of the min and max, given code 0, and written to the block's
// table as rows by token: row pointers (entries of the tokens before t),
// then the entries in flat-index order (an entry's place is the number of
// selected indices below its own).
//
// write_kernel: widens new sink tokens to fp32 (tract #2458, sink commit) and
// copies new tokens into the fp16 ring at slot (a - S) mod R (pigeon guide,
// step 4).  It runs after flush_kernel on the same stream, because a flush can
// read ring slots that the write then overwrites.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kFlushThreads = 256;

// Group grp of unit (bb, h): the body of both flush kernels.  Shared memory:
// keys [G][d] fp16, values [G][d] fp16, key codes [G][d] u8, value codes
// [G][d] u8, the per-thread key (min, max) of its share of a channel (2 x
// kFlushThreads floats); with outliers also the key and value flag bitmasks
// (G d / 32 words each), the selected flat indices of keys and values (n_out
// each) and the round maxima (2 x 8 words).
size_t flush_smem(const Geo& g) {
  const size_t gd = static_cast<size_t>(g.G) * g.d;
  size_t s = gd * (2 * sizeof(__half) + 2) + 2 * kFlushThreads * sizeof(float);
  if (g.n_out > 0) s += 2 * (gd / 32) * 4 + 2 * static_cast<size_t>(g.n_out) * 4 + 16 * 4;
  return s;
}

// the largest key below prev over the block's n elements of x; every thread
// gets it (one barrier per call; red alternates between two halves by round)
__device__ __forceinline__ uint32_t block_next_key(const __half* x, int n, uint32_t prev, uint32_t* red, int round) {
  uint32_t best = 0u;
  const unsigned short* xb = reinterpret_cast<const unsigned short*>(x);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t k = (static_cast<uint32_t>(xb[i] & 0x7FFFu) << 16) | (0xFFFFu - static_cast<uint32_t>(i));
    if (k < prev && k > best) best = k;
  }
  best = __reduce_max_sync(0xffffffffu, best);
  uint32_t* rr = red + 8 * (round & 1);
  if ((threadIdx.x & 31) == 0) rr[threadIdx.x >> 5] = best;
  __syncthreads();
  uint32_t m = 0u;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = rr[w] > m ? rr[w] : m;
  return m;
}

// selects the n_out outliers of a [G][d] block x: flags them in f (zeroed
// here) and writes the table at out: row pointers by token, then from
// out_ent the entries in flat-index order; sel is scratch for n_out indices.
// Ends with a barrier: the flags are then visible to all.
__device__ __forceinline__ void select_outliers(const __half* x, int G, int d, int n_out, int out_ent, uint32_t* f,
                                                int* sel, uint32_t* red, uint8_t* out) {
  const int n = G * d;
  for (int w = threadIdx.x; w < n / 32; w += blockDim.x) f[w] = 0u;
  uint32_t prev = 0xFFFFFFFFu;
  for (int r = 0; r < n_out; ++r) {
    prev = block_next_key(x, n, prev, red, r);
    if (threadIdx.x == 0) sel[r] = static_cast<int>(0xFFFFu - (prev & 0xFFFFu));
  }
  __syncthreads();
  const unsigned short* xb = reinterpret_cast<const unsigned short*>(x);
  uint32_t* table = reinterpret_cast<uint32_t*>(out + out_ent);
  uint16_t* ptr = reinterpret_cast<uint16_t*>(out);
  for (int t = threadIdx.x; t <= G; t += blockDim.x) {   // entries of the tokens before t
    int cnt = 0;
    for (int j = 0; j < n_out; ++j) cnt += sel[j] < t * d ? 1 : 0;
    ptr[t] = static_cast<uint16_t>(cnt);
  }
  for (int e = threadIdx.x; e < n_out; e += blockDim.x) {
    const int i = sel[e];
    int rank = 0;
    for (int j = 0; j < n_out; ++j) rank += sel[j] < i ? 1 : 0;
    atomicOr(&f[i >> 5], 1u << (i & 31));
    // {u8 t, u8 c, fp16 x}, little-endian
    table[rank] = static_cast<uint32_t>(i / d) | (static_cast<uint32_t>(i % d) << 8) |
                  (static_cast<uint32_t>(xb[i]) << 16);
  }
  __syncthreads();
}

__device__ __forceinline__ bool flagged(const uint32_t* f, int i) { return (f[i >> 5] >> (i & 31)) & 1u; }

// rintf(__fdiv_rn(a, dq)) for 0 <= a <= max - min, dq the fp16-rounded
// (max - min) / (2^b - 1) and rq = __frcp_rn(dq).  Rounding to nearest keeps
// dq at least half of the unrounded step, so the exact quotient Q = a / dq
// is below 512.  The product q = RN(a rq) lies within Q 2^-23 <= 2^-14 of Q
// and the division's RN(Q) within 2^-16, so q and RN(Q) are less than 2^-13
// apart and round to the same integer unless q lies within 2^-11 of a
// half-integer; there the division itself is done.
__device__ __forceinline__ float code_of(float a, float dq, float rq) {
  float q = __fmul_rn(a, rq);
  if (fabsf(q - floorf(q) - 0.5f) < 0x1p-11f) q = __fdiv_rn(a, dq);
  return rintf(q);
}

__device__ __forceinline__ void flush_group(const Geo& g, uint8_t* __restrict__ arena,
                                            const __half* __restrict__ k_new, const __half* __restrict__ v_new,
                                            int64_t T_old, int64_t n_stride, int64_t grp, int h, int bb) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = g.G, d = g.d, b = g.bits;
  __half* kx = reinterpret_cast<__half*>(smem);
  __half* vx = kx + G * d;
  uint8_t* kc = reinterpret_cast<uint8_t*>(vx + G * d);
  uint8_t* vc = kc + G * d;
  float* kmn = reinterpret_cast<float*>(vc + G * d);   // [kFlushThreads]: a thread's share of a channel
  float* kmx = kmn + kFlushThreads;

  uint8_t* unit = arena + (static_cast<int64_t>(bb) * g.hkv + h) * g.unit_bytes;
  const int64_t in_off = (static_cast<int64_t>(bb) * g.hkv + h) * n_stride * d;   // input row of (bb, h)
  const int64_t a0 = g.S + grp * G;

  // stage the group's tokens: 16-byte chunks of each d-wide row
  const int chunks = d / 8;
  for (int i = threadIdx.x; i < G * chunks; i += blockDim.x) {
    const int t = i / chunks, c8 = (i % chunks) * 8;
    const int64_t a = a0 + t;
    const __half* ks;
    const __half* vs;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (a < T_old) {
      const int64_t slot = (a - g.S) % g.R;
      ks = reinterpret_cast<const __half*>(unit + g.res_k) + slot * d;
      vs = reinterpret_cast<const __half*>(unit + g.res_v) + slot * d;
      if (dbg_in_region(g, ks + c8, 16) && dbg_in_region(g, vs + c8, 16)) {
        kv = *reinterpret_cast<const uint4*>(ks + c8);
        vv = *reinterpret_cast<const uint4*>(vs + c8);
      }
    } else {
      ks = k_new + in_off + (a - T_old) * d;
      vs = v_new + in_off + (a - T_old) * d;
      kv = *reinterpret_cast<const uint4*>(ks + c8);
      vv = *reinterpret_cast<const uint4*>(vs + c8);
      dbg_check_finite(g, kv);
      dbg_check_finite(g, vv);
    }
    *reinterpret_cast<uint4*>(kx + t * d + c8) = kv;
    *reinterpret_cast<uint4*>(vx + t * d + c8) = vv;
  }
  __syncthreads();

  const float top = static_cast<float>((1 << b) - 1);
  uint8_t* blk = unit + g.groups + (grp % g.n_slots) * g.block_bytes;
  if (!dbg_in_region(g, blk, g.block_bytes)) return;   // uniform over the block
  __half* ks_out = reinterpret_cast<__half*>(blk + g.blk_ks);
  __half* vs_out = reinterpret_cast<__half*>(blk + g.blk_vs);

  // outliers: flags (bit t d + c) of the key and value blocks
  const bool outl = g.n_out > 0;
  uint32_t* kf = reinterpret_cast<uint32_t*>(kmx + kFlushThreads);
  uint32_t* vf = kf + G * d / 32;
  if (outl) {
    int* sel = reinterpret_cast<int*>(vf + G * d / 32);
    uint32_t* red = reinterpret_cast<uint32_t*>(sel + g.n_out);
    select_outliers(kx, G, d, g.n_out, g.out_ent, kf, sel, red, blk + g.blk_ko);
    select_outliers(vx, G, d, g.n_out, g.out_ent, vf, sel, red, blk + g.blk_vo);
  }

  // keys: one (Δ, min) per channel over the group's tokens (its dense values).
  // The block's threads split each channel's tokens into np parts (thread
  // part * d + c takes channel c, tokens [part G / np, (part + 1) G / np)),
  // whose minima and maxima meet in shared memory
  const int np = static_cast<int>(blockDim.x) / d;   // 2 at d = 128, 4 at d = 64
  const int kc_ch = static_cast<int>(threadIdx.x) % d, kpart = static_cast<int>(threadIdx.x) / d;
  const bool kthread = kpart < np;
  const int kt0 = kpart * G / np, kt1 = (kpart + 1) * G / np;
  if (kthread) {
    float mn = INFINITY, mx = -INFINITY;
    for (int t = kt0; t < kt1; ++t) {
      if (outl && flagged(kf, t * d + kc_ch)) continue;
      const float v = __half2float(kx[t * d + kc_ch]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    kmn[threadIdx.x] = mn;
    kmx[threadIdx.x] = mx;
  }
  __syncthreads();
  if (kthread) {
    const int c = kc_ch;
    float mn = INFINITY, mx = -INFINITY;
    for (int p2 = 0; p2 < np; ++p2) {
      mn = fminf(mn, kmn[p2 * d + c]);
      mx = fmaxf(mx, kmx[p2 * d + c]);
    }
    if (mn > mx) { mn = 0.0f; mx = 0.0f; }   // every value an outlier
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    const __half d16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), top));
    const float dq = __half2float(d16);
    const float rq = dq != 0.0f ? __frcp_rn(dq) : 0.0f;
    for (int t = kt0; t < kt1; ++t) {
      int code = 0;
      if (dq != 0.0f && !(outl && flagged(kf, t * d + c))) {
        const float r = code_of(__fsub_rn(__half2float(kx[t * d + c]), mn), dq, rq);
        code = static_cast<int>(fminf(fmaxf(r, 0.0f), top));
      }
      kc[t * d + c] = static_cast<uint8_t>(code);
    }
    if (kpart == 0) {
      ks_out[c] = d16;
      ks_out[d + c] = __float2half_rn(mn);
    }
  }

  // values: one (Δ, min) per token over the channels; one warp per token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int t = warp; t < G; t += nwarps) {
    float mn = INFINITY, mx = -INFINITY;
    for (int c = lane; c < d; c += 32) {
      if (outl && flagged(vf, t * d + c)) continue;
      const float v = __half2float(vx[t * d + c]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (mn > mx) { mn = 0.0f; mx = 0.0f; }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    const __half d16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), top));
    const float dq = __half2float(d16);
    const float rq = dq != 0.0f ? __frcp_rn(dq) : 0.0f;
    for (int c = lane; c < d; c += 32) {
      int code = 0;
      if (dq != 0.0f && !(outl && flagged(vf, t * d + c))) {
        const float r = code_of(__fsub_rn(__half2float(vx[t * d + c]), mn), dq, rq);
        code = static_cast<int>(fminf(fmaxf(r, 0.0f), top));
      }
      vc[t * d + c] = static_cast<uint8_t>(code);
    }
    if (lane == 0) {
      vs_out[2 * t] = d16;
      vs_out[2 * t + 1] = __float2half_rn(mn);
    }
  }
  __syncthreads();

  if (!(b == 2 || b == 4 || b == 8)) {
    // the other widths: a bit stream per row, code j at bits [b j, b j + b);
    // one thread per output byte
    const int krow = d * b / 8, vrow = G * b / 8;
    uint8_t* kq8 = blk + g.blk_kq;
    for (int i = threadIdx.x; i < G * krow; i += blockDim.x) {
      const int t = i / krow, byte = i % krow;
      uint32_t v = 0;
      for (int k = 0; k < 8; ++k) {
        const int bit = 8 * byte + k, j = bit / b;
        v |= ((static_cast<uint32_t>(kc[t * d + j]) >> (bit - j * b)) & 1u) << k;
      }
      kq8[i] = static_cast<uint8_t>(v);
    }
    uint8_t* vq8 = blk + g.blk_vq;
    for (int i = threadIdx.x; i < d * vrow; i += blockDim.x) {
      const int c = i / vrow, byte = i % vrow;
      uint32_t v = 0;
      for (int k = 0; k < 8; ++k) {
        const int bit = 8 * byte + k, j = bit / b;
        v |= ((static_cast<uint32_t>(vc[j * d + c]) >> (bit - j * b)) & 1u) << k;
      }
      vq8[i] = static_cast<uint8_t>(v);
    }
    return;
  }
  // pack: element j of a 32-bit word goes to half (j & 1), bit b * (j >> 1)
  const int per = 32 / b;
  uint32_t* kq = reinterpret_cast<uint32_t*>(blk + g.blk_kq);
  const int kwords = G * (d / per);            // key rows: G tokens x d channels
  for (int i = threadIdx.x; i < kwords; i += blockDim.x) {
    const int t = i / (d / per), w = i % (d / per);
    uint32_t word = 0;
    for (int j = 0; j < per; ++j)
      word |= static_cast<uint32_t>(kc[t * d + w * per + j]) << (16 * (j & 1) + b * (j >> 1));
    kq[i] = word;
  }
  uint32_t* vq = reinterpret_cast<uint32_t*>(blk + g.blk_vq);
  const int vwords = d * (G / per);            // value rows: d channels x G tokens
  for (int i = threadIdx.x; i < vwords; i += blockDim.x) {
    const int c = i / (G / per), w = i % (G / per);
    uint32_t word = 0;
    for (int j = 0; j < per; ++j)
      word |= static_cast<uint32_t>(vc[(w * per + j) * d + c]) << (16 * (j & 1) + b * (j >> 1));
    vq[i] = word;
  }
}

__global__ void __launch_bounds__(kFlushThreads)
flush_kernel(Geo g, uint8_t* __restrict__ arena, const __half* __restrict__ k_new,
             const __half* __restrict__ v_new, int64_t T_old, int64_t n_stride, int64_t g_begin) {
  flush_group(g, arena, k_new, v_new, T_old, n_stride, g_begin + blockIdx.x, blockIdx.y, blockIdx.z);
}

// The fused step over a ragged batch: block (h, b) freezes sequence b's next
// group if its new token (position T_old of its run) reaches a full ring.
__global__ void __launch_bounds__(kFlushThreads)
flush_ragged_kernel(Geo g, uint8_t* __restrict__ arena, const __half* __restrict__ k_new,
                    const __half* __restrict__ v_new, const __grid_constant__ RunTable rt) {
  const int bb = blockIdx.z;
  int k = 0;
  while (k < rt.n && bb >= rt.r[k].b0 + rt.r[k].nb) ++k;
  if (k == rt.n || bb < rt.r[k].b0) return;   // not in this launch's runs (uniform per block)
  const int64_t T_old = rt.r[k].fresh_pos;
  const State s0 = state_at(g, T_old), s1 = state_at(g, T_old + 1);
  if (s1.n_groups == s0.n_groups) return;   // uniform per block
  flush_group(g, arena, k_new, v_new, T_old, 1, s0.n_groups, blockIdx.y, bb);
}

// One thread per 8 channels of one token of one unit.
__global__ void write_kernel(Geo g, uint8_t* __restrict__ arena, const __half* __restrict__ k_new,
                             const __half* __restrict__ v_new, int64_t T_old, int64_t n_new,
                             int64_t n_stride, int64_t sink_end, int64_t ring_begin) {
  const int d = g.d, chunks = d / 8;
  const int64_t n_sink_new = sink_end > T_old ? sink_end - T_old : 0;
  const int64_t n_ring_new = T_old + n_new - ring_begin;
  const int64_t per_unit = (n_sink_new + n_ring_new) * chunks;
  const int64_t total = per_unit * g.B * g.hkv;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t u = i / per_unit, r = i % per_unit;
    const int64_t k = r / chunks;
    const int c8 = static_cast<int>(r % chunks) * 8;
    const int64_t a = (k < n_sink_new) ? T_old + k : ring_begin + (k - n_sink_new);
    const int64_t src = (u * n_stride + (a - T_old)) * d + c8;
    uint8_t* unit = arena + u * g.unit_bytes;
    const uint4 kv = *reinterpret_cast<const uint4*>(k_new + src);
    const uint4 vv = *reinterpret_cast<const uint4*>(v_new + src);
    dbg_check_finite(g, kv);
    dbg_check_finite(g, vv);
    if (a < g.S) {
      const __half2* kh = reinterpret_cast<const __half2*>(&kv);
      const __half2* vh = reinterpret_cast<const __half2*>(&vv);
      float* sk = reinterpret_cast<float*>(unit + g.sink_k) + a * d + c8;
      float* sv = reinterpret_cast<float*>(unit + g.sink_v) + a * d + c8;
      if (!dbg_in_region(g, sk, 32) || !dbg_in_region(g, sv, 32)) continue;
      float2 f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = __half22float2(kh[j]);
      reinterpret_cast<float4*>(sk)[0] = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
      reinterpret_cast<float4*>(sk)[1] = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = __half22float2(vh[j]);
      reinterpret_cast<float4*>(sv)[0] = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
      reinterpret_cast<float4*>(sv)[1] = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
    } else {
      const int64_t slot = (a - g.S) % g.R;
      __half* rk = reinterpret_cast<__half*>(unit + g.res_k) + slot * d + c8;
      __half* rv = reinterpret_cast<__half*>(unit + g.res_v) + slot * d + c8;
      if (!dbg_in_region(g, rk, 16) || !dbg_in_region(g, rv, 16)) continue;
      *reinterpret_cast<uint4*>(rk) = kv;
      *reinterpret_cast<uint4*>(rv) = vv;
    }
  }
}

}  // namespace

cudaError_t launch_flush(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_stride, int64_t g_begin, int64_t g_end,
                         cudaStream_t stream) {
  if (g_end <= g_begin) return cudaSuccess;
  const size_t smem = flush_smem(g);
  cudaError_t e = cudaFuncSetAttribute(flush_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int64_t left = g_end - g_begin;
  int64_t start = g_begin;
  while (left > 0) {   // grid.x is limited to 2^31-1; chunk for safety
    const int64_t n = left < 65535 * 256 ? left : 65535 * 256;
    dim3 grid(static_cast<unsigned>(n), g.hkv, g.B);
    if (injected_launch_failure()) return cudaErrorLaunchFailure;
    flush_kernel<<<grid, kFlushThreads, smem, stream>>>(g, arena, k_new, v_new, T_old, n_stride, start);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    start += n;
    left -= n;
  }
  return cudaSuccess;
}

cudaError_t launch_flush_ragged(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                                const RunTable& runs, cudaStream_t stream) {
  const size_t smem = flush_smem(g);
  cudaError_t e = cudaFuncSetAttribute(flush_ragged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  flush_ragged_kernel<<<dim3(1, g.hkv, g.B), kFlushThreads, smem, stream>>>(g, arena, k_new, v_new, runs);
  return cudaGetLastError();
}

cudaError_t launch_write(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_new, int64_t n_stride, int64_t ring_begin, cudaStream_t stream) {
  const int64_t T_new = T_old + n_new;
  const int64_t sink_end = T_new < g.S ? T_new : g.S;
  const int64_t n_sink_new = sink_end > T_old ? sink_end - T_old : 0;
  const int64_t n_ring_new = T_new - ring_begin;
  const int64_t total = (n_sink_new + n_ring_new) * (g.d / 8) * g.B * g.hkv;
  if (total <= 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  write_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(g, arena, k_new, v_new, T_old, n_new,
                                                                       n_stride, sink_end, ring_begin);
  return cudaGetLastError();
}

}  // namespace kivi
