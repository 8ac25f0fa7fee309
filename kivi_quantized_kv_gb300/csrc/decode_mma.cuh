// decode_mma.cuh — tensor-core split-K decode attention over the packed cache.
//
// softmax(q Kᵀ / sqrt(d)) V with K and V dequantized group by group on the
// fly and no fp16 copy in memory (KV-cache quantization guide (pigeon), "How
// it works", step 5); the query heads of a GQA group share one pass over their
// kv head (tract #2329, "What's in the PR").
//
// Work split (stream-K).  A "unit" is one (sequence, kv head, head pass); a
// head pass covers up to four query heads.  Unit u owns `uw` work positions:
// its visible frozen groups, then `tc` positions that stand for its tail (the
// fp32 sinks and the fp16 ring).  The units' positions, laid end to end, are
// cut into one equal contiguous range per CTA, and the grid is one wave of
// resident CTAs, so every SM gets the same work and none idles.  A CTA walks
// the units its range touches; for each it processes the groups in its range
// (warp w: the range's groups w, w + nw, ...) and, if its range holds the
// unit's first tail position, the whole tail.
//
// Frozen groups:
//  * every group block (codes + scales, one contiguous range) is copied
//    HBM -> shared memory by one 1-D cp.async.bulk completing on an mbarrier;
//    a warp keeps `ns` blocks in flight and keeps issuing into the next unit
//    of its range while it finishes the current one;
//  * codes become exact fp16 values with one AND: a b-bit code c masked into
//    an fp16 word with a zero exponent is the subnormal c * 2^-24 (times 2^k
//    for a field at bit k of its half), which the tensor cores multiply
//    exactly; 2^-k goes into the other operand and 2^24 into the result;
//  * scores: mma.sync m16n8k16 with A = key codes (16 tokens x 16 channels)
//    and B = the folded query q_c Δ_c split exactly into hi = fp16(q Δ) and
//    lo = q Δ - hi in two columns per head, so every product is exact and the
//    fp32 accumulation is as good as an fp32 dot product; a second MMA adds
//    Σ_c q_c min_c (q·k̂_t = Σ_c (q_c Δ_c) code_tc + Σ_c q_c min_c exactly);
//  * online softmax in log2 units, rescaled only when the running max grows
//    by more than 2^8 (the stale max keeps every p <= 256);
//  * values: Oᵀ += Vᵀ P' with A = value codes (16 channels x 16 tokens: a
//    channel's tokens are contiguous in the block) and B = p_t Δ_t split into
//    hi/lo fp16; P' moves from the score layout to the B layout through a
//    512-byte per-warp shared buffer; Σ_t p_t min_t is added per head.
// Tails: a warp takes 32 tokens at a time; for q·k each lane owns a token and
// reads its whole row, for P·V each lane owns D/32 consecutive channels and
// the probabilities are broadcast by shuffles; fp32 throughout.
// Epilogue of every unit a CTA touches: the CTA combines its warps in shared
// memory; a unit covered by one CTA is written out directly, otherwise each
// CTA writes its partial (o, m, l) and the last CTA of the unit to finish (a
// per-unit counter) merges all partials and resets the counter.
#pragma once

#include "kivi_internal.cuh"

#include <math.h>

namespace kivi {
namespace mma {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;                         // lazy rescale threshold (log2 units)
constexpr unsigned long long kWaitNs = 2000000000ull;    // bounded wait on a copy: 2 s
constexpr float kTwo24 = 16777216.0f;                    // codes enter the MMAs scaled by 2^-24

struct Args {
  Geo g;
  const uint8_t* arena;
  const __half* q;
  __half* out;
  float* partials;      // [B][h_q][stride][d + 2]
  unsigned* counters;   // [units]: CTAs finished per unit
  unsigned* error;      // bit 0: a copy wait timed out
  DecodePlan plan;
  int32_t ns;           // copy stages per warp
  int32_t stage_bytes;  // bytes per stage (block bytes rounded up to 128)
  int32_t stride;       // partial records per (sequence, query head)
  int32_t npass;        // head passes per kv head
  int32_t units;        // B * h_kv * npass
  int32_t tc;           // work positions standing for one tail
  int64_t uw;           // work positions per unit: visible groups + tc
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arms the barrier for `bytes` of copies (one arrival).
__device__ __forceinline__ void bulk_arm(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One bulk copy global -> shared that completes `bytes` on the barrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  bulk_arm(bar, bytes);
  bulk_copy(dst, src, bytes, bar);
}

// A tail chunk: the sinks in chunks of 4 fp32 tokens, then the ring in chunks
// of 8 fp16 tokens; in a stage, keys at offset 0 and values at 16 * D bytes.
constexpr int kSinkChunk = 4;
constexpr int kRingChunk = 8;
struct TailChunk {
  int sink;        // 1 = fp32 sink rows
  int n;           // tokens in the chunk (0 only when the cache is empty)
  int first;       // first sink index, or first ring token (0-based, oldest first)
};
__device__ __forceinline__ TailChunk tail_chunk(int idx, int n_sink, int n_res) {
  TailChunk t;
  const int n_sc = (n_sink + kSinkChunk - 1) / kSinkChunk;
  if (idx < n_sc) {
    t.sink = 1;
    t.first = idx * kSinkChunk;
    t.n = min(kSinkChunk, n_sink - t.first);
  } else {
    t.sink = 0;
    t.first = (idx - n_sc) * kRingChunk;
    t.n = max(0, min(kRingChunk, n_res - t.first));
  }
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for a barrier phase; gives up after kWaitNs and reports false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));   // low half = lo
  return r;
}

// Bit position (within its 16-bit half) of element pair p of a lane's row
// slice: the packing puts element j of a 32-bit word in half j & 1 at bit
// BITS*(j >> 1), so pair p = elements (2p, 2p + 1) sits at the same bit of
// both halves.  8-bit pairs are moved to bit 0 by a byte permute.
template <int BITS>
__host__ __device__ constexpr int pair_bit(int p) {
  return BITS == 8 ? 0 : BITS * ((p % (16 / BITS)) % (8 / BITS));
}

// fp16x2 of pair p as exact subnormals: low half = element 2p, high half =
// element 2p + 1, each code * 2^(pair_bit(p) - 24).
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* w, int p) {
  if constexpr (BITS == 8) {
    // bytes (p&1) and (p&1)+2 of the word into the low byte of each half
    return prmt(w[p >> 1], 0u, (p & 1) ? 0x4341u : 0x4240u);
  } else {
    constexpr int PPW = 16 / BITS;   // pairs per word
    constexpr int PPB = 8 / BITS;    // pairs per byte position
    const int pp = p % PPW;
    const uint32_t x = w[p / PPW] >> (8 * (pp / PPB));
    return x & (((1u << BITS) - 1u) * (0x00010001u << pair_bit<BITS>(p)));
  }
}

// fp16x2 with both halves 2^-k (k in {0, 2, 4, 6}).
__host__ __device__ constexpr uint32_t pow2_neg_h2(int k) {
  return k == 0 ? 0x3C003C00u : k == 2 ? 0x34003400u : k == 4 ? 0x2C002C00u : 0x24002400u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// CTA that owns work position x when W positions are cut into P ranges
// [floor(c W / P), floor((c + 1) W / P)).
__device__ __forceinline__ int owner_of(int64_t x, int64_t W, int64_t P) {
  const int64_t c = ((x + 1) * P - 1) / W;
  return static_cast<int>(c < P - 1 ? c : P - 1);
}

template <int D, int BITS, int CH>
__global__ void __launch_bounds__(256, 2) decode_mma_kernel(const Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr int RK = D * BITS / 8;          // key row bytes
  constexpr int KW = RK / 16;               // 32-bit words of a lane's key quarter
  constexpr int NKC = D / 16;               // k-chunks over channels
  constexpr int QV = CH * BITS / 4;         // bits of a lane's value quarter per chunk of CH tokens
  constexpr int VW = QV >= 32 ? QV / 32 : 1;
  constexpr int TPL = CH / 8;               // tokens per score lane per chunk
  constexpr int NCT = D / 16;               // channel tiles
  constexpr int NKT = CH / 16;              // token k-chunks per chunk (value MMA)
  constexpr int NC = D / 32;                // channels per lane in the tail

  const Geo& g = a.g;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int rep = g.rep;
  const int64_t T = a.plan.st.T;
  const int64_t lo_pos = g.window > 0 ? T - g.window : INT64_MIN;
  const float qscale = kLog2e * rsqrtf(static_cast<float>(D));
  const int64_t n_vis = a.plan.n_vis_groups;
  const int64_t P = gridDim.x;
  const int64_t W = static_cast<int64_t>(a.units) * a.uw;
  const int64_t c_start = (static_cast<int64_t>(blockIdx.x) * W) / P;
  const int64_t c_end = (static_cast<int64_t>(blockIdx.x + 1) * W) / P;
  if (c_start >= c_end) return;   // uniform; only when W < P, which the host avoids
  const int u_first = static_cast<int>(c_start / a.uw);
  const int u_last = static_cast<int>((c_end - 1) / a.uw);

  // shared memory: stages | red_m, red_l, red_o | merge weights | q (tail, fp32) | q (fp16) | exchange | barriers
  uint8_t* stages = smem_raw;
  float* red_m = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(nw) * a.ns * a.stage_bytes);
  float* red_l = red_m + nw * 4;
  float* red_o = red_l + nw * 4;
  float* mrg = red_o + nw * 4 * D;                  // [4][stride] merge weights
  float* qs = mrg + 4 * a.stride;                    // [4][D + 4] scaled q of the tail
  __half* qh_s = reinterpret_cast<__half*>(qs + 4 * (D + 4));   // [4][D] q of the unit's heads (0 past nh)
  __half* xchg = qh_s + 4 * D;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xchg + nw * 8 * CH);
  __shared__ unsigned s_last;

  uint8_t* my_stages = stages + static_cast<size_t>(warp) * a.ns * a.stage_bytes;
  const uint32_t bar0 = smem_addr(bars + warp * a.ns);
  __half* xw = xchg + warp * 8 * CH;
  const uint32_t blk_bytes = static_cast<uint32_t>(g.block_bytes);

  if (lane == 0) {
    for (int s = 0; s < a.ns; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // group positions [lo, hi) of unit u inside this CTA's range
  auto seg_groups = [&](int u, int64_t& lo, int64_t& hi) {
    const int64_t base = static_cast<int64_t>(u) * a.uw;
    lo = (c_start > base ? c_start : base) - base;
    hi = (c_end < base + a.uw ? c_end : base + a.uw) - base;
    if (lo > n_vis) lo = n_vis;
    if (hi > n_vis) hi = n_vis;
  };
  auto warp_count = [&](int64_t lo, int64_t hi) -> int {
    return (lo + warp < hi) ? static_cast<int>((hi - lo - warp + nw - 1) / nw) : 0;
  };
  auto unit_base = [&](int u) -> const uint8_t* {
    const int per_b = g.hkv * a.npass;
    const int bb = u / per_b, hk = (u % per_b) / a.npass;
    return a.arena + (static_cast<int64_t>(bb) * g.hkv + hk) * g.unit_bytes;
  };

  // per-warp copy pipeline over the warp's work positions of the whole range
  // (group blocks and tail chunks alike); the producer (lane 0) walks units
  // lazily, so per issued block it only adds
  const uint32_t n_slots = static_cast<uint32_t>(g.n_slots);
  const bool ring_slots = g.window > 0;
  const int t_sink = static_cast<int>(a.plan.st.n_sink), t_res = static_cast<int>(a.plan.st.n_res);
  const int rs0 = static_cast<int>((a.plan.st.n_groups * g.G) % g.R);   // ring slot of the oldest ring token
  int c_st = 0;                 // consumer: stage, phase parity
  uint32_t c_ph = 0;
  int inflight = 0;             // blocks issued and not yet consumed
  int p_st = 0;                 // producer: next stage
  int pu = u_first;             // producer: unit being issued
  int p_left = -1;              // positions of unit pu this warp still has to issue (-1: not entered)
  int64_t p_pos = 0;            // next position (unit-local)
  const uint8_t* p_unit = nullptr;
  bool aborted = false;
  auto produce = [&]() {
    if (lane != 0 || aborted) return;
    while (inflight < a.ns) {
      if (p_left <= 0) {
        if (p_left == 0) ++pu;
        if (pu > u_last) return;
        const int64_t base = static_cast<int64_t>(pu) * a.uw;
        const int64_t lo = (c_start > base ? c_start : base) - base;
        const int64_t hi = (c_end < base + a.uw ? c_end : base + a.uw) - base;
        p_left = warp_count(lo, hi);
        p_pos = lo + warp;
        p_unit = unit_base(pu);
        if (p_left == 0) continue;
      }
      const uint32_t dst = smem_addr(my_stages + p_st * a.stage_bytes);
      const uint32_t bar = bar0 + 8 * p_st;
      bool issued = true;
      if (p_pos < n_vis) {   // a frozen group block
        const uint32_t grp = static_cast<uint32_t>(a.plan.g_first + p_pos);
        const uint32_t slot = ring_slots ? grp % n_slots : grp;
        bulk_load(dst, p_unit + g.groups + static_cast<int64_t>(slot) * g.block_bytes, blk_bytes, bar);
      } else {                // a tail chunk: key rows then value rows
        const TailChunk tk = tail_chunk(static_cast<int>(p_pos - n_vis), t_sink, t_res);
        if (tk.n == 0) {
          issued = false;
        } else if (tk.sink) {
          const uint32_t bytes = static_cast<uint32_t>(tk.n) * D * 4;
          bulk_arm(bar, 2 * bytes);
          bulk_copy(dst, p_unit + g.sink_k + static_cast<int64_t>(tk.first) * D * 4, bytes, bar);
          bulk_copy(dst + 16 * D, p_unit + g.sink_v + static_cast<int64_t>(tk.first) * D * 4, bytes, bar);
        } else {
          int s0 = rs0 + tk.first;
          if (s0 >= g.R) s0 -= g.R;
          const int n1 = min(tk.n, g.R - s0), n2 = tk.n - n1;   // the ring may wrap
          bulk_arm(bar, static_cast<uint32_t>(tk.n) * D * 4);
          bulk_copy(dst, p_unit + g.res_k + static_cast<int64_t>(s0) * D * 2, n1 * D * 2, bar);
          bulk_copy(dst + 16 * D, p_unit + g.res_v + static_cast<int64_t>(s0) * D * 2, n1 * D * 2, bar);
          if (n2 > 0) {
            bulk_copy(dst + n1 * D * 2, p_unit + g.res_k, n2 * D * 2, bar);
            bulk_copy(dst + 16 * D + n1 * D * 2, p_unit + g.res_v, n2 * D * 2, bar);
          }
        }
      }
      if (issued) {
        if (++p_st == a.ns) p_st = 0;
        ++inflight;
      }
      p_pos += nw;
      --p_left;
    }
  };

  const uint32_t partmask = (r & 1) ? 0xFFFFFFFFu : 0u;   // B column r: head r >> 1, lo part if odd
  const int hh_col = r >> 1;

  for (int u = u_first; u <= u_last; ++u) {
    const int per_b = g.hkv * a.npass;
    const int ub = u / per_b, uh = (u % per_b) / a.npass, upass = u % a.npass;
    const int h0 = upass * 4;
    const int nh = min(4, rep - h0);
    const uint8_t* unit = unit_base(u);
    int64_t glo, ghi;
    seg_groups(u, glo, ghi);
    const int n_mine = warp_count(glo, ghi);
    const int64_t ubase = static_cast<int64_t>(u) * a.uw;
    // positions of this unit in the CTA's range; those past n_vis are tail
    // chunks of 32 sink/ring tokens, dealt to the warps round-robin like groups
    const int64_t lo_full = (c_start > ubase ? c_start : ubase) - ubase;
    const int64_t hi_full = (c_end < ubase + a.uw ? c_end : ubase + a.uw) - ubase;
    const int64_t tlo = lo_full > n_vis ? lo_full : n_vis;
    const bool do_tail = tlo < hi_full;   // CTA-uniform
    int64_t my_tail = hi_full;            // this warp's first tail position
    if (do_tail) {
      const int64_t off = (tlo - lo_full) % nw;
      my_tail = tlo + (warp - off + nw) % nw;
    }
    const int first = owner_of(ubase, W, P);
    const int total = owner_of(ubase + a.uw - 1, W, P) - first + 1;
    const int slot = static_cast<int>(blockIdx.x) - first;

    // the unit's query heads, once per unit for all warps: fp16 [4][D] for the
    // tensor cores (zero past nh), fp32 [D][4] scaled for the tail
    {
      const __half* qsrc = a.q + (static_cast<int64_t>(ub) * g.hq + uh * rep + h0) * D;
      for (int i = threadIdx.x; i < 4 * D / 8; i += blockDim.x) {
        const int hh = i / (D / 8), c8 = (i % (D / 8)) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (hh < nh) v = __ldg(reinterpret_cast<const uint4*>(qsrc + hh * D + c8));
        *reinterpret_cast<uint4*>(qh_s + hh * D + c8) = v;
      }
      if (do_tail) {   // [4][D + 4]: padded rows keep the four heads in different banks
        for (int i = threadIdx.x; i < 4 * D; i += blockDim.x) {
          const int hh = i / D, ch = i % D;
          qs[hh * (D + 4) + ch] = (hh < nh) ? __half2float(qsrc[hh * D + ch]) * qscale : 0.f;
        }
      }
      __syncthreads();
    }

    float res_m = -INFINITY, res_l = 0.f, res_mn = 0.f;
    float oacc[NCT][4];
#pragma unroll
    for (int i = 0; i < NCT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    if (n_mine > 0) {
      // ---------------------------------------------------------- frozen groups
      // this lane's B column r = (head r >> 1, part r & 1), channel quarter c
      const __half* qlane = qh_s + hh_col * D + c * (D / 4);
      for (int t = 0; t < n_mine; ++t) {
        produce();
        __syncwarp();
        if (aborted) continue;
        const int st = c_st;
        if (!mbar_wait(bar0 + 8 * st, c_ph)) {
          aborted = true;
          if (lane == 0) atomicOr(a.error, 1u);
          continue;
        }
        const int64_t grp = a.plan.g_first + glo + warp + static_cast<int64_t>(t) * nw;
        const uint8_t* blk = my_stages + st * a.stage_bytes;

        // (1) folded query B fragments: hi = fp16(q Δ) in even columns, lo = q Δ - hi in
        // odd ones, times 2^-k for the bit position k of the key code pair they multiply
        uint32_t q2[NKC][2];
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const uint4 v = reinterpret_cast<const uint4*>(qlane)[i];
          q2[2 * i][0] = v.x; q2[2 * i][1] = v.y; q2[2 * i + 1][0] = v.z; q2[2 * i + 1][1] = v.w;
        }
        uint32_t bq[NKC][2];
        const uint8_t* ks = blk + g.blk_ks;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const uint4 dv = *reinterpret_cast<const uint4*>(ks + c * (D / 2) + 16 * i);
          const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int kcn = 2 * i + (j >> 1), sl = j & 1;
            const uint32_t hi = hmul2_u(q2[kcn][sl], dw[j]);
            uint32_t v = hfma2_u(q2[kcn][sl], dw[j], (hi ^ 0x80008000u) & partmask);
            const int kb = pair_bit<BITS>(2 * kcn + sl);
            if (kb != 0) v = hmul2_u(v, pow2_neg_h2(kb));
            bq[kcn][sl] = v;
          }
        }
        // (2) Σ_c q_c min_c for every head (hi columns), one MMA per k-chunk
        float cst[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const uint4 mv = *reinterpret_cast<const uint4*>(ks + 2 * D + c * (D / 2) + 16 * i);
          const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
          for (int v2 = 0; v2 < 2; ++v2) {
            const int kcn = 2 * i + v2;
            mma16816(cst, mw[2 * v2], mw[2 * v2], mw[2 * v2 + 1], mw[2 * v2 + 1], q2[kcn][0] & ~partmask,
                     q2[kcn][1] & ~partmask);
          }
        }
        const float cst_h = cst[0] * qscale;
        const float sc_scale = qscale * kTwo24;
        const __half* vsc = reinterpret_cast<const __half*>(blk + g.blk_vs);
        const int64_t a_grp = g.S + grp * g.G;

        for (int s0 = 0; s0 < g.G; s0 += CH) {
          // (3) scores: lane (r, c) gets head c's scores of tokens s0 + TPL*r + i
          float sv[TPL];
#pragma unroll
          for (int v2 = 0; v2 < TPL / 2; ++v2) {
            uint32_t w0[KW], w1[KW];
            // 64-byte rows: odd r takes the pair's rows in swapped order so the
            // two rows of a shared-memory phase fall in different bank halves
            constexpr bool kSwap = (RK == 64);
            const int sw = kSwap ? (r & 1) : 0;
            const uint8_t* row0 = blk + g.blk_kq + (s0 + TPL * r + 2 * v2 + sw) * RK + c * (RK / 4);
            const uint8_t* row1 = blk + g.blk_kq + (s0 + TPL * r + 2 * v2 + 1 - sw) * RK + c * (RK / 4);
            if constexpr (KW >= 4) {
#pragma unroll
              for (int i = 0; i < KW; i += 4) {
                const uint4 x = *reinterpret_cast<const uint4*>(row0 + 4 * i);
                const uint4 y = *reinterpret_cast<const uint4*>(row1 + 4 * i);
                w0[i] = x.x; w0[i + 1] = x.y; w0[i + 2] = x.z; w0[i + 3] = x.w;
                w1[i] = y.x; w1[i + 1] = y.y; w1[i + 2] = y.z; w1[i + 3] = y.w;
              }
            } else if constexpr (KW == 2) {
              const uint2 x = *reinterpret_cast<const uint2*>(row0);
              const uint2 y = *reinterpret_cast<const uint2*>(row1);
              w0[0] = x.x; w0[1] = x.y; w1[0] = y.x; w1[1] = y.y;
            } else {
              w0[0] = *reinterpret_cast<const uint32_t*>(row0);
              w1[0] = *reinterpret_cast<const uint32_t*>(row1);
            }
            // two accumulators halve the dependent MMA chain
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kcn = 0; kcn < NKC; ++kcn) {
              if (kcn & 1) {
                mma16816(acd, code_pair<BITS>(w0, 2 * kcn), code_pair<BITS>(w1, 2 * kcn),
                         code_pair<BITS>(w0, 2 * kcn + 1), code_pair<BITS>(w1, 2 * kcn + 1), bq[kcn][0], bq[kcn][1]);
              } else {
                mma16816(acc, code_pair<BITS>(w0, 2 * kcn), code_pair<BITS>(w1, 2 * kcn),
                         code_pair<BITS>(w0, 2 * kcn + 1), code_pair<BITS>(w1, 2 * kcn + 1), bq[kcn][0], bq[kcn][1]);
              }
            }
            const float s_a = fmaf((acc[0] + acc[1]) + (acd[0] + acd[1]), sc_scale, cst_h);
            const float s_b = fmaf((acc[2] + acc[3]) + (acd[2] + acd[3]), sc_scale, cst_h);
            sv[2 * v2] = sw ? s_b : s_a;
            sv[2 * v2 + 1] = sw ? s_a : s_b;
          }
          if (g.window > 0) {   // tokens before T - W are invisible
#pragma unroll
            for (int i = 0; i < TPL; ++i)
              if (a_grp + s0 + TPL * r + i < lo_pos) sv[i] = -INFINITY;
          }
          // (4) online softmax for head c, lazy rescale
          float mx = sv[0];
#pragma unroll
          for (int i = 1; i < TPL; ++i) mx = fmaxf(mx, sv[i]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          if (mx > res_m + kRescale) {   // uniform over the 8 lanes of head c
            const float corr = (res_m == -INFINITY) ? 0.f : exp2f(res_m - mx);
            res_m = mx;
            res_l *= corr;
            res_mn *= corr;
#pragma unroll
            for (int i = 0; i < NCT; ++i) { oacc[i][0] *= corr; oacc[i][1] *= corr; oacc[i][2] *= corr; oacc[i][3] *= corr; }
          }
          float pd[TPL];
          {
            const __half2* vp = reinterpret_cast<const __half2*>(vsc) + s0 + TPL * r;
#pragma unroll
            for (int i = 0; i < TPL; ++i) {
              const float2 dm = __half22float2(vp[i]);
              const float p = (res_m == -INFINITY) ? 0.f : exp2f(sv[i] - res_m);
              res_l += p;
              res_mn = fmaf(p, dm.y, res_mn);
              pd[i] = p * dm.x;
            }
          }
          // (5) P' hi/lo into the exchange buffer: row 2c = hi, 2c + 1 = lo
          {
            uint32_t hw[TPL / 2], lw[TPL / 2];
#pragma unroll
            for (int i = 0; i < TPL / 2; ++i) {
              const float a0 = pd[2 * i], a1 = pd[2 * i + 1];
              const float h0f = __uint_as_float(__float_as_uint(a0) & 0xFFFFE000u);
              const float h1f = __uint_as_float(__float_as_uint(a1) & 0xFFFFE000u);
              hw[i] = (c < nh) ? pack_half2(h0f, h1f) : 0u;
              lw[i] = (c < nh) ? pack_half2(a0 - h0f, a1 - h1f) : 0u;
            }
            uint32_t* xh = reinterpret_cast<uint32_t*>(xw + (2 * c) * CH + TPL * r);
            uint32_t* xl = reinterpret_cast<uint32_t*>(xw + (2 * c + 1) * CH + TPL * r);
#pragma unroll
            for (int i = 0; i < TPL / 2; ++i) { xh[i] = hw[i]; xl[i] = lw[i]; }
          }
          __syncwarp();
          // (6) Oᵀ += Vᵀ P': B = P' of tokens c*CH/4 + 4kc + {0,1 | 2,3} in column r,
          // times 2^-k for the bit position of the value code pair
          uint32_t bp[NKT][2];
#pragma unroll
          for (int kcn = 0; kcn < NKT; ++kcn) {
            const uint2 x = *reinterpret_cast<const uint2*>(xw + r * CH + c * (CH / 4) + 4 * kcn);
            const int k0 = pair_bit<BITS>(2 * kcn), k1 = pair_bit<BITS>(2 * kcn + 1);
            bp[kcn][0] = k0 ? hmul2_u(x.x, pow2_neg_h2(k0)) : x.x;
            bp[kcn][1] = k1 ? hmul2_u(x.y, pow2_neg_h2(k1)) : x.y;
          }
          const uint8_t* vq = blk + g.blk_vq + s0 * BITS / 8;
#pragma unroll
          for (int ct = 0; ct < NCT; ++ct) {
            uint32_t v0[VW], v1[VW];
            const uint8_t* rowa = vq + static_cast<int64_t>(16 * ct + r) * (g.G * BITS / 8);
            const uint8_t* rowb = rowa + 8 * (g.G * BITS / 8);
            if constexpr (QV >= 32) {
#pragma unroll
              for (int i = 0; i < VW; ++i) {
                v0[i] = reinterpret_cast<const uint32_t*>(rowa + c * (QV / 8))[i];
                v1[i] = reinterpret_cast<const uint32_t*>(rowb + c * (QV / 8))[i];
              }
            } else {
              const int bitpos = c * QV;
              const int sh = (bitpos % 32) / 2;
              v0[0] = reinterpret_cast<const uint32_t*>(rowa)[bitpos / 32] >> sh;
              v1[0] = reinterpret_cast<const uint32_t*>(rowb)[bitpos / 32] >> sh;
            }
#pragma unroll
            for (int kcn = 0; kcn < NKT; ++kcn) {
              mma16816(oacc[ct], code_pair<BITS>(v0, 2 * kcn), code_pair<BITS>(v1, 2 * kcn),
                       code_pair<BITS>(v0, 2 * kcn + 1), code_pair<BITS>(v1, 2 * kcn + 1), bp[kcn][0], bp[kcn][1]);
            }
          }
          __syncwarp();
        }
        // stage released; produce() refills it on the next step
        if (++c_st == a.ns) { c_st = 0; c_ph ^= 1u; }
        --inflight;
      }
    }

    // group state -> reduction slot `warp`
    {
      float lh = res_l, mh = res_mn;
      lh += __shfl_xor_sync(0xffffffffu, lh, 4);
      lh += __shfl_xor_sync(0xffffffffu, lh, 8);
      lh += __shfl_xor_sync(0xffffffffu, lh, 16);
      mh += __shfl_xor_sync(0xffffffffu, mh, 4);
      mh += __shfl_xor_sync(0xffffffffu, mh, 8);
      mh += __shfl_xor_sync(0xffffffffu, mh, 16);
      if (c < nh) {
        if (r == 0) {
          red_m[warp * 4 + c] = res_m;
          red_l[warp * 4 + c] = lh;
        }
        float* ro = red_o + (warp * 4 + c) * D;
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct) {
          ro[16 * ct + r] = fmaf(oacc[ct][0] + oacc[ct][1], kTwo24, mh);
          ro[16 * ct + r + 8] = fmaf(oacc[ct][2] + oacc[ct][3], kTwo24, mh);
        }
      }
    }

    // ------------------------------------------------------------------ tail
    // this warp's tail chunks (sinks, then ring), from the copy stages, folded
    // into its reduction slot
    if (my_tail < hi_full) {
      float t_m[4], t_l[4], t_o[4][NC];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        t_m[hh] = -INFINITY; t_l[hh] = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j) t_o[hh][j] = 0.f;
      }
      const int tt = lane >> 2, th = lane & 3;   // q·k lanes: (token, head)
      for (int64_t pos_t = my_tail; pos_t < hi_full; pos_t += nw) {
        produce();
        __syncwarp();
        const TailChunk tk = tail_chunk(static_cast<int>(pos_t - n_vis), t_sink, t_res);
        if (tk.n == 0 || aborted) continue;
        const int st = c_st;
        if (!mbar_wait(bar0 + 8 * st, c_ph)) {
          aborted = true;
          if (lane == 0) atomicOr(a.error, 1u);
          continue;
        }
        const uint8_t* kst = my_stages + st * a.stage_bytes;
        const uint8_t* vst = kst + 16 * D;
        // scores: lane (token tt, head th)
        float sc = -INFINITY;
        if (tt < tk.n && th < nh) {
          const float* qrow = qs + th * (D + 4);
          float acc = 0.f;
          if (tk.sink) {
            const float* kr = reinterpret_cast<const float*>(kst) + tt * D;
#pragma unroll 8
            for (int c4 = 0; c4 < D / 4; ++c4) {
              const float4 kk = reinterpret_cast<const float4*>(kr)[c4];
              const float4 qq = reinterpret_cast<const float4*>(qrow)[c4];
              acc = fmaf(qq.x, kk.x, acc); acc = fmaf(qq.y, kk.y, acc);
              acc = fmaf(qq.z, kk.z, acc); acc = fmaf(qq.w, kk.w, acc);
            }
          } else {
            const __half* kr = reinterpret_cast<const __half*>(kst) + tt * D;
#pragma unroll 4
            for (int c8 = 0; c8 < D / 8; ++c8) {
              const uint4 kk = reinterpret_cast<const uint4*>(kr)[c8];
              const __half2* kh = reinterpret_cast<const __half2*>(&kk);
              const float4 qa = reinterpret_cast<const float4*>(qrow)[2 * c8];
              const float4 qb = reinterpret_cast<const float4*>(qrow)[2 * c8 + 1];
              float2 f;
              f = __half22float2(kh[0]); acc = fmaf(qa.x, f.x, acc); acc = fmaf(qa.y, f.y, acc);
              f = __half22float2(kh[1]); acc = fmaf(qa.z, f.x, acc); acc = fmaf(qa.w, f.y, acc);
              f = __half22float2(kh[2]); acc = fmaf(qb.x, f.x, acc); acc = fmaf(qb.y, f.y, acc);
              f = __half22float2(kh[3]); acc = fmaf(qb.z, f.x, acc); acc = fmaf(qb.w, f.y, acc);
            }
          }
          sc = acc;
        }
        // per-head max and sum over the chunk (lanes of one head differ in bits 2..4)
        float mx = sc;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        float mnew[4], corr[4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          mnew[hh] = fmaxf(t_m[hh], __shfl_sync(0xffffffffu, mx, hh));
          corr[hh] = (t_m[hh] == -INFINITY) ? 0.f : exp2f(t_m[hh] - mnew[hh]);
        }
        const float mine = (th == 0) ? mnew[0] : (th == 1) ? mnew[1] : (th == 2) ? mnew[2] : mnew[3];
        const float pv = (sc == -INFINITY) ? 0.f : exp2f(sc - mine);
        float ps = pv;
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          t_l[hh] = t_l[hh] * corr[hh] + __shfl_sync(0xffffffffu, ps, hh);
          t_m[hh] = mnew[hh];
#pragma unroll
          for (int j = 0; j < NC; ++j) t_o[hh][j] *= corr[hh];
        }
        // P·V: lane owns channels lane*NC ..; p of (token t, head hh) sits in lane 4t + hh
        for (int t = 0; t < tk.n; ++t) {
          float vv[NC];
          if (tk.sink) {
            const float* vr = reinterpret_cast<const float*>(vst) + t * D + lane * NC;
            if constexpr (NC == 4) {
              const float4 x = *reinterpret_cast<const float4*>(vr);
              vv[0] = x.x; vv[1] = x.y; vv[2] = x.z; vv[3] = x.w;
            } else {
              const float2 x = *reinterpret_cast<const float2*>(vr);
              vv[0] = x.x; vv[1] = x.y;
            }
          } else {
            const __half* vr = reinterpret_cast<const __half*>(vst) + t * D + lane * NC;
            if constexpr (NC == 4) {
              const uint2 x = *reinterpret_cast<const uint2*>(vr);
              const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
              const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
              vv[0] = f0.x; vv[1] = f0.y; vv[2] = f1.x; vv[3] = f1.y;
            } else {
              const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(vr));
              vv[0] = f0.x; vv[1] = f0.y;
            }
          }
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            const float pw = __shfl_sync(0xffffffffu, pv, 4 * t + hh);
#pragma unroll
            for (int j = 0; j < NC; ++j) t_o[hh][j] = fmaf(pw, vv[j], t_o[hh][j]);
          }
        }
        __syncwarp();
        if (++c_st == a.ns) { c_st = 0; c_ph ^= 1u; }
        --inflight;
      }
      // merge into the warp's slot: M = max(m_g, m_t), both sides rescaled
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float l = t_l[hh];   // already summed over the warp
        if (hh < nh) {
          const float mg = red_m[warp * 4 + hh], lg = red_l[warp * 4 + hh];
          const float M = fmaxf(mg, t_m[hh]);
          const float fg = (mg == -INFINITY) ? 0.f : exp2f(mg - M);
          const float ft = (t_m[hh] == -INFINITY) ? 0.f : exp2f(t_m[hh] - M);
          float* ro = red_o + (warp * 4 + hh) * D + lane * NC;
#pragma unroll
          for (int j = 0; j < NC; ++j) ro[j] = ro[j] * fg + t_o[hh][j] * ft;
          __syncwarp();
          if (lane == 0) {
            red_m[warp * 4 + hh] = M;
            red_l[warp * 4 + hh] = lg * fg + l * ft;
          }
        }
      }
    }
    __syncthreads();

    // ---------------------------------------------------------- epilogue
    const int64_t head0 = static_cast<int64_t>(ub) * g.hq + uh * rep + h0;
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
      const int hh = i / D, ch = i % D;
      float M = -INFINITY;
      for (int w = 0; w < nw; ++w) M = fmaxf(M, red_m[w * 4 + hh]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < nw; ++w) {
          const float mw = red_m[w * 4 + hh];
          if (mw == -INFINITY) continue;
          const float f = exp2f(mw - M);
          L = fmaf(red_l[w * 4 + hh], f, L);
          O = fmaf(red_o[(w * 4 + hh) * D + ch], f, O);
        }
      }
      if (total == 1) {
        a.out[(head0 + hh) * D + ch] = __float2half_rn(L > 0.f ? O / L : 0.f);
      } else {
        float* dst = a.partials + ((head0 + hh) * a.stride + slot) * (D + 2);
        dst[ch] = O;
        if (ch == 0) { dst[D] = M; dst[D + 1] = L; }
      }
    }
    if (total > 1) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) s_last = (atomicAdd(a.counters + u, 1u) == static_cast<unsigned>(total - 1)) ? 1u : 0u;
      __syncthreads();
      if (s_last) {
        // merge every partial of this unit: M = max m_s, w_s = 2^(m_s - M),
        // L = Σ l_s w_s, out = Σ o_s w_s / L
        __threadfence();
        for (int i = threadIdx.x; i < nh * total; i += blockDim.x) {
          const int hh = i / total, s = i % total;
          mrg[hh * a.stride + s] = __ldcg(a.partials + ((head0 + hh) * a.stride + s) * (D + 2) + D);
        }
        __syncthreads();
        if (threadIdx.x < nh) {
          const int hh = threadIdx.x;
          float M = -INFINITY;
          for (int s = 0; s < total; ++s) M = fmaxf(M, mrg[hh * a.stride + s]);
          red_m[hh] = M;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nh * total; i += blockDim.x) {
          const int hh = i / total, s = i % total;
          const float M = red_m[hh], ms = mrg[hh * a.stride + s];
          mrg[hh * a.stride + s] = (M == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - M);
        }
        __syncthreads();
        if (threadIdx.x < nh) {
          const int hh = threadIdx.x;
          float L = 0.f;
          for (int s = 0; s < total; ++s)
            L = fmaf(__ldcg(a.partials + ((head0 + hh) * a.stride + s) * (D + 2) + D + 1), mrg[hh * a.stride + s], L);
          red_l[hh] = L;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
          const int hh = i / D, ch = i % D;
          const float* basep = a.partials + (head0 + hh) * a.stride * (D + 2) + ch;
          const float* wgt = mrg + hh * a.stride;
          float O = 0.f;
#pragma unroll 8
          for (int s = 0; s < total; ++s) O = fmaf(__ldcg(basep + s * (D + 2)), wgt[s], O);
          const float L = red_l[hh];
          a.out[(head0 + hh) * D + ch] = __float2half_rn(L > 0.f ? O / L : 0.f);
        }
        if (threadIdx.x == 0) a.counters[u] = 0u;
      }
    }
    __syncthreads();
  }

  // drain this warp's copies still in flight (only after an abort), bounded
  if (aborted) {
    for (int k = 0; k < inflight; ++k) {
      mbar_wait(bar0 + 8 * c_st, c_ph);
      if (++c_st == a.ns) { c_st = 0; c_ph ^= 1u; }
    }
  }
}

}  // namespace mma
}  // namespace kivi
