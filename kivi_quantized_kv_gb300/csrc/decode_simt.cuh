// decode_simt.cuh — split-K decode attention on CUDA cores for the code widths
// packed as a plain bit stream (b in {1, 3, 5, 6, 7}; tract #2329 makes the
// width configurable, the kvquant++ README recommends 3 bits) at head dim 64.
//
// The tensor-core kernel (decode_mma.cuh) reads a lane's quarter of a key
// row as whole 32-bit words; at head dim 64 a quarter of a bit-stream row is
// 16 b bits, which does not start on a word for odd b.  These shapes
// dequantize on CUDA cores instead, each lane owning whole rows, in fp32:
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
//
// Pre-RoPE keys (ROPE; pigeon guide, "KVQuant adds": keys quantized before
// the rotary embedding, which would otherwise mix channel pairs): the codes
// hold the unrotated keys, and every dequantized key is rotated at its own
// position a before the dot product, pairs (i, i + D/2) by the angle
// a θ_i, θ_i = base^(-2i/D); the query arrives rotated.  A per-token
// rotation does not fold into one operand shared by a group's tokens, so
// these caches decode here, at every code width.  cos and sin of a θ_i:
//   * frozen groups, a = a0 + t: angle addition of the group's base a0 θ_i
//     (one per pair and group, from a double-precision angle reduced mod 2π)
//     and the offset t θ_i (a per-CTA table [D/2][G], built once);
//   * sinks and ring tokens: the double-precision angle of each token.
// The score of token t for a head, with k_i = min_i + code_i Δ_i:
//   s = Σ_i cos (k_i q_i + k_{i+D/2} q_{i+D/2}) + sin (k_i q_{i+D/2} - k_{i+D/2} q_i).
#pragma once

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
// Shared memory of one warp: two block buffers (the copy of the next group
// overlaps the current one's arithmetic), then floats: q of every head (for
// tails), q Δ of every head (per group), p Δ or p (values).
template <int D>
struct Smem {
  __host__ __device__ static int block_bytes(const Geo& g) { return static_cast<int>((g.block_bytes + 15) / 16 * 16); }
  __host__ __device__ static int bytes(const Geo& g) {
    return 2 * block_bytes(g) + 4 * (2 * kMaxRep * D + kMaxRep * 64);
  }
};

// 32 codes of BITS bits held in BITS consecutive 32-bit words, as floats.
// Bit-stream widths: code j at bit BITS j of the words taken as one
// little-endian bit string.  Widths 2, 4, 8 (the word rule): word j / (32 /
// BITS) holds code j at bit 16 (e & 1) + BITS (e >> 1), e = j mod (32 / BITS).
// Every shift is a compile-time constant.
template <int BITS>
__device__ __forceinline__ void unpack32(const uint32_t (&w)[BITS], float (&f)[32]) {
  constexpr uint32_t M = (1u << BITS) - 1u;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    uint32_t v;
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
      constexpr int per = 32 / BITS;
      const int e = j % per;
      v = (w[j / per] >> (16 * (e & 1) + BITS * (e >> 1))) & M;
    } else {
      const int bit = BITS * j, wi = bit >> 5, sh = bit & 31;
      if (sh + BITS <= 32) v = (w[wi] >> sh) & M;
      else v = __funnelshift_r(w[wi], w[wi + 1], sh) & M;
    }
    f[j] = static_cast<float>(v);
  }
}

// code j of a packed row (the same packing as unpack32), with run-time shifts
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t* row, int j) {
  constexpr uint32_t M = (1u << BITS) - 1u;
  if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
    constexpr int per = 32 / BITS;
    const int e = j % per;
    return (row[j / per] >> (16 * (e & 1) + BITS * (e >> 1))) & M;
  } else {
    const int bit = BITS * j, wi = bit >> 5, sh = bit & 31;
    uint32_t v = row[wi] >> sh;
    if (sh + BITS > 32) v |= row[wi + 1] << (32 - sh);
    return v & M;
  }
}

// cos and sin of a double-precision angle, reduced mod 2π in double first
// (positions times θ reach 10^5 rad), then taken in single precision
__device__ __forceinline__ float2 rope_cs(double ang) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  const double r = ang - kTwoPi * rint(ang * (1.0 / kTwoPi));
  float sn, cs;
  sincosf(static_cast<float>(r), &sn, &cs);
  return make_float2(cs, sn);
}

// shared memory of the RoPE tables of one CTA: θ (double) [D/2], the offset
// table [D/2][G] and one base row [D/2] per warp (float2)
__host__ __device__ inline int rope_bytes(const Geo& g) {
  const int h = g.d / 2;
  return g.rope_l2b != 0.0 ? h * 8 + h * g.G * 8 + kWarps * h * 8 : 0;
}

// 16-byte asynchronous copies global -> shared (Ampere-style cp.async; the
// group is waited for with cp.async.wait_group)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

template <int D, int BITS, bool ROPE>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(const Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int H2 = D / 2;
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
  const int bbytes = Smem<D>::block_bytes(g);
  float* qs = reinterpret_cast<float*>(my + 2 * bbytes);               // [rep][D] q * qscale
  float* qd = qs + kMaxRep * D;                                        // [rep][D] q Δ * qscale
  float* pv = qd + kMaxRep * D;                                        // [rep][64] p Δ or p

  // q of the unit's heads, scaled to log2 units
  for (int i = lane; i < rep * D; i += 32) {
    const int h = i / D, c = i % D;
    qs[i] = __half2float(a.q[(static_cast<int64_t>(bb) * g.hq + hk * rep + h) * D + c]) * qscale;
  }
  __syncwarp();

  // RoPE tables: θ_i, the offsets' cos / sin, this warp's base row
  double* theta = reinterpret_cast<double*>(smem + kWarps * Smem<D>::bytes(g));
  float2* offs = reinterpret_cast<float2*>(theta + H2);          // [H2][G]
  float2* wbase = offs + H2 * g.G + warp * H2;                   // [H2]
  if constexpr (ROPE) {
    for (int i = threadIdx.x; i < H2; i += blockDim.x) theta[i] = exp2(-(2.0 * i / D) * g.rope_l2b);
    __syncthreads();
    for (int x = threadIdx.x; x < H2 * g.G; x += blockDim.x)
      offs[x] = rope_cs(static_cast<double>(x % g.G) * theta[x / g.G]);
    __syncthreads();
  }

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

  // the copy of item `it` (a frozen group) into buffer `buf`
  auto prefetch = [&](int it, int buf) {
    if (it >= i1 || it >= n_vis) return;
    const int64_t grp = a.plan.g_first + it;
    const int64_t slot = g.window > 0 ? grp % g.n_slots : grp;
    const uint8_t* src = ubase + g.groups + slot * g.block_bytes;
    uint8_t* dst = my + buf * bbytes;
    for (int i = lane; i < static_cast<int>(g.block_bytes / 16); i += 32) cp_async16(dst + 16 * i, src + 16 * i);
  };
  constexpr int KW = D / 32;   // 32-channel chunks of a key row
  int buf = 0;
  prefetch(i0 + warp, 0);
  cp_async_commit();
  for (int it = i0 + warp; it < i1; it += kWarps) {
    prefetch(it + kWarps, buf ^ 1);   // the next item's copy runs under this one's arithmetic
    cp_async_commit();
    if (it < n_vis) {
      // ------------------------------------------------ a frozen group
      cp_async_wait<1>();   // this item's copy (the older group) has landed
      __syncwarp();
      const uint8_t* blk = my + buf * bbytes;
      const int64_t grp = a.plan.g_first + it;
      const __half* ks = reinterpret_cast<const __half*>(blk + g.blk_ks);   // Δ[D], min[D]
      const __half* vs = reinterpret_cast<const __half*>(blk + g.blk_vs);   // (Δ, min) per token
      // q Δ per head and channel; Σ q min per head (without RoPE)
      float cmin[kMaxRep];
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) cmin[h] = 0.f;
      for (int c = lane; c < (ROPE ? 0 : D); c += 32) {
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
      for (int h = 0; h < kMaxRep; ++h) {
        if (h >= rep) break;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cmin[h] += __shfl_xor_sync(0xffffffffu, cmin[h], off);
      }
      __syncwarp();
      const int64_t a0 = g.S + grp * G;
      const int ns = G / 32;   // tokens per lane (G in {32, 64})
      if constexpr (ROPE) {   // the group's base angles a0 θ_i
        for (int i = lane; i < H2; i += 32) wbase[i] = rope_cs(static_cast<double>(a0) * theta[i]);
        __syncwarp();
      }
      // scores: lane = token t = lane + 32 i; each 32-channel chunk of its
      // row is unpacked once and used by every head
      float s[2][kMaxRep];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= ns) break;
        const int t = lane + 32 * i;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(blk + g.blk_kq + t * (D * BITS / 8));
        float acc[kMaxRep];
        if constexpr (ROPE) {
          // the pairs (i, i + D/2): codes read one at a time (a rolled loop
          // keeps the registers and the code small), dequantized, rotated at
          // position a0 + t, dotted with every head's q
#pragma unroll
          for (int h = 0; h < kMaxRep; ++h) acc[h] = 0.f;
#pragma unroll 2
          for (int ci = 0; ci < H2; ++ci) {
            const float k1 = fmaf(static_cast<float>(code_at<BITS>(row, ci)), __half2float(ks[ci]),
                                  __half2float(ks[D + ci]));
            const float k2 = fmaf(static_cast<float>(code_at<BITS>(row, ci + H2)), __half2float(ks[ci + H2]),
                                  __half2float(ks[D + ci + H2]));
            const float2 b = wbase[ci], o = offs[ci * G + t];
            const float cs = b.x * o.x - b.y * o.y, sn = b.y * o.x + b.x * o.y;
            const float r1 = k1 * cs - k2 * sn, r2 = k2 * cs + k1 * sn;
#pragma unroll
            for (int h = 0; h < kMaxRep; ++h) {
              if (h >= rep) break;
              acc[h] = fmaf(qs[h * D + ci], r1, fmaf(qs[h * D + ci + H2], r2, acc[h]));
            }
          }
        } else {
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) acc[h] = cmin[h];
#pragma unroll
        for (int k = 0; k < KW; ++k) {
          uint32_t w[BITS];
#pragma unroll
          for (int x = 0; x < BITS; ++x) w[x] = row[k * BITS + x];
          float f[32];
          unpack32<BITS>(w, f);
#pragma unroll
          for (int h = 0; h < kMaxRep; ++h) {
            if (h >= rep) break;
            const float4* qh = reinterpret_cast<const float4*>(qd + h * D + 32 * k);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float4 qv = qh[x];
              acc[h] = fmaf(qv.x, f[4 * x], acc[h]);
              acc[h] = fmaf(qv.y, f[4 * x + 1], acc[h]);
              acc[h] = fmaf(qv.z, f[4 * x + 2], acc[h]);
              acc[h] = fmaf(qv.w, f[4 * x + 3], acc[h]);
            }
          }
        }
        }
        const bool vis = a0 + t >= lo_pos;
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) s[i][h] = vis ? acc[h] : -INFINITY;
      }
      // softmax per head; p Δ_t into shared memory; Σ_t p_t min_t
      float pmin[kMaxRep];
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        pmin[h] = 0.f;
        if (h >= rep) break;
        float sh[2] = {s[0][h], ns > 1 ? s[1][h] : -INFINITY}, p[2] = {0.f, 0.f};
        softmax(h, sh, p, ns);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= ns) break;
          const int t = lane + 32 * i;
          const float vd = __half2float(vs[2 * t]), vm = __half2float(vs[2 * t + 1]);
          pv[h * 64 + t] = p[i] * vd;
          pmin[h] = fmaf(p[i], vm, pmin[h]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) pmin[h] += __shfl_xor_sync(0xffffffffu, pmin[h], off);
      }
      __syncwarp();
      // values: lane = channel c = lane + 32 j; each 32-token chunk of its row
      // is unpacked once and used by every head
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(blk + g.blk_vq + c * (G * BITS / 8));
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          if (h >= rep) break;
          o[h][j] += pmin[h];
        }
        for (int k = 0; k < ns; ++k) {
          uint32_t w[BITS];
#pragma unroll
          for (int x = 0; x < BITS; ++x) w[x] = row[k * BITS + x];
          float f[32];
          unpack32<BITS>(w, f);
#pragma unroll
          for (int h = 0; h < kMaxRep; ++h) {
            if (h >= rep) break;
            const float4* ph = reinterpret_cast<const float4*>(pv + h * 64 + 32 * k);
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float4 pq = ph[x];
              acc = fmaf(pq.x, f[4 * x], acc);
              acc = fmaf(pq.y, f[4 * x + 1], acc);
              acc = fmaf(pq.z, f[4 * x + 2], acc);
              acc = fmaf(pq.w, f[4 * x + 3], acc);
            }
            o[h][j] += acc;
          }
        }
      }
      __syncwarp();
    } else {
      // ------------------------------------------------ a tail chunk of up to 32 tokens
      const int tc = it - n_vis;
      const bool sink = tc < a.sink_items;
      const int first = sink ? kTail * tc : kTail * (tc - a.sink_items);
      const int n = sink ? min(kTail, n_sink - first) : min(kTail, n_res - first);
      if (n <= 0) { buf ^= 1; continue; }
      // token u of the chunk: its key and value rows are read whole by the
      // warp (lane = channel lane + 32 j, coalesced); scores by a warp sum
      auto kval = [&](int u, int c) -> float {
        if (sink) return reinterpret_cast<const float*>(ubase + g.sink_k)[static_cast<int64_t>(first + u) * D + c];
        const int slot = (rs0 + first + u) % g.R;
        return __half2float(reinterpret_cast<const __half*>(ubase + g.res_k)[static_cast<int64_t>(slot) * D + c]);
      };
      auto vval = [&](int u, int c) -> float {
        if (sink) return reinterpret_cast<const float*>(ubase + g.sink_v)[static_cast<int64_t>(first + u) * D + c];
        const int slot = (rs0 + first + u) % g.R;
        return __half2float(reinterpret_cast<const __half*>(ubase + g.res_v)[static_cast<int64_t>(slot) * D + c]);
      };
      // every sink and ring token lies inside any window (W >= R): no mask
      float sc[kMaxRep];   // lane u keeps token u's score of every head
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) sc[h] = -INFINITY;
      for (int u = 0; u < n; ++u) {
        float kr[CPL];
#pragma unroll
        for (int jj = 0; jj < CPL; ++jj) kr[jj] = kval(u, lane + 32 * jj);
        if constexpr (ROPE) {   // channels lane + 32 jj and their partners + D/2, at the token's position
          const int64_t pos = sink ? static_cast<int64_t>(first + u)
                                   : g.S + a.plan.st.n_groups * g.G + first + u;
#pragma unroll
          for (int jj = 0; jj < CPL / 2; ++jj) {
            const float2 r = rope_cs(static_cast<double>(pos) * theta[lane + 32 * jj]);
            const float x = kr[jj], y = kr[jj + CPL / 2];
            kr[jj] = x * r.x - y * r.y;
            kr[jj + CPL / 2] = y * r.x + x * r.y;
          }
        }
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          if (h >= rep) break;
          float part = 0.f;
#pragma unroll
          for (int jj = 0; jj < CPL; ++jj) part = fmaf(qs[h * D + lane + 32 * jj], kr[jj], part);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
          if (lane == u) sc[h] = part;
        }
      }
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        if (h >= rep) break;
        float sh[2] = {sc[h], -INFINITY}, p[2] = {0.f, 0.f};
        softmax(h, sh, p, 1);
        pv[h * 64 + lane] = p[0];
      }
      __syncwarp();
      for (int u = 0; u < n; ++u) {
#pragma unroll
        for (int jj = 0; jj < CPL; ++jj) {
          const float v = vval(u, lane + 32 * jj);
#pragma unroll
          for (int h = 0; h < kMaxRep; ++h) {
            if (h >= rep) break;
            o[h][jj] = fmaf(pv[h * 64 + u], v, o[h][jj]);
          }
        }
      }
      __syncwarp();
    }
    buf ^= 1;
  }
  cp_async_wait<0>();

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

// Launches a.splits CTAs per unit; with `resident` non-null it only reports
// the CTAs of this instantiation one SM holds at `smem`.
template <int D, int BITS, bool ROPE>
cudaError_t launch_one(const Args& a, int ctas, int smem, cudaStream_t s, int* resident) {
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<D, BITS, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  if (resident)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(resident, decode_simt_kernel<D, BITS, ROPE>, kWarps * 32, smem);
  decode_simt_kernel<D, BITS, ROPE><<<ctas, kWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// with RoPE: every width (decode_simt_rope_d{64,128}.cu)
template <int D>
cudaError_t launch_rope_d(const Args& a, int ctas, int smem, cudaStream_t s, int* resident) {
  switch (a.g.bits) {
    case 1: return launch_one<D, 1, true>(a, ctas, smem, s, resident);
    case 2: return launch_one<D, 2, true>(a, ctas, smem, s, resident);
    case 3: return launch_one<D, 3, true>(a, ctas, smem, s, resident);
    case 4: return launch_one<D, 4, true>(a, ctas, smem, s, resident);
    case 5: return launch_one<D, 5, true>(a, ctas, smem, s, resident);
    case 6: return launch_one<D, 6, true>(a, ctas, smem, s, resident);
    case 7: return launch_one<D, 7, true>(a, ctas, smem, s, resident);
    case 8: return launch_one<D, 8, true>(a, ctas, smem, s, resident);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_rope_d64(const Args& a, int ctas, int smem, cudaStream_t s, int* resident);
cudaError_t launch_rope_d128(const Args& a, int ctas, int smem, cudaStream_t s, int* resident);

// without RoPE: the bit-stream widths
template <int D>
cudaError_t launch_d(const Args& a, int ctas, int smem, cudaStream_t s, int* resident) {
  if (a.g.rope_l2b != 0.0)
    return D == 64 ? launch_rope_d64(a, ctas, smem, s, resident) : launch_rope_d128(a, ctas, smem, s, resident);
  switch (a.g.bits) {
    case 1: return launch_one<D, 1, false>(a, ctas, smem, s, resident);
    case 3: return launch_one<D, 3, false>(a, ctas, smem, s, resident);
    case 5: return launch_one<D, 5, false>(a, ctas, smem, s, resident);
    case 6: return launch_one<D, 6, false>(a, ctas, smem, s, resident);
    case 7: return launch_one<D, 7, false>(a, ctas, smem, s, resident);
    default: return cudaErrorInvalidValue;
  }
}

// defined in decode_simt_d64.cu and decode_simt_d128.cu
cudaError_t launch_d64(const Args& a, int ctas, int smem, cudaStream_t s, int* resident);
cudaError_t launch_d128(const Args& a, int ctas, int smem, cudaStream_t s, int* resident);

}  // namespace simt
}  // namespace kivi
