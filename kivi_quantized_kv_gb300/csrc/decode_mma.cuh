// decode_mma.cuh — tensor-core split-K decode attention over the packed cache.
//
// softmax(q Kᵀ / sqrt(d)) V with K and V dequantized group by group on the
// fly and no fp16 copy in memory (KV-cache quantization guide (pigeon), "How
// it works", step 5); the query heads of a GQA group share one pass over their
// kv head (tract #2329, "What's in the PR").
//
// Work split (stream-K).  A "unit" is one (sequence, kv head, head pass); a
// head pass covers up to four query rows.  The rows of a kv head are its
// query heads times the query tokens: nq = 1 for a decode, and nq = M for the
// causal attention of a chunk's M newest tokens, where row v is query token
// v / rep (position q_pos0 + v / rep) of head v % rep of the GQA group, and
// each row sees only the tokens at or before its position (and, with a
// window, within the W tokens ending there).  Unit u owns `uw` work positions:
// its visible frozen groups, then `tc` positions for its tail (the fp32 sinks
// in chunks of 4 tokens, then the fp16 ring in chunks of 8).  The units'
// positions, laid end to end, are cut into one equal contiguous range per CTA,
// and the grid is one wave of resident CTAs.  Inside a CTA the warps claim
// the range's positions two at a time from a shared counter (one at a time
// near the range's end), so a warp that is held up (say, by combining a
// unit) simply takes fewer, and the warps finish close together.
//
// Warps never wait for one another while they stream:
//  * each warp runs its own copy pipeline: lane 0 claims a position, issues
//    one 1-D cp.async.bulk per item into the warp's next stage (completing on
//    that stage's mbarrier) and keeps `ns` items in flight, walking on into
//    the next unit while the warp still computes the current one.  Before
//    its first position of a unit a warp copies the unit's query rows (so no
//    CTA barrier is needed to share them);
//  * a warp that finishes a unit leaves its (m, l, o) in its shared-memory
//    slot and signs in; the last warp of the CTA to sign in combines the
//    slots, writes the output (unit inside one CTA) or the CTA's partial, and
//    bumps the unit's counter; the last CTA of the unit merges the partials.
//    The other warps go straight on; a slot is rewritten only after the
//    previous combine has read it (a generation count, bounded wait).
//
// Frozen groups:
//  * codes become exact fp16 values with one AND: a b-bit code c masked into
//    an fp16 word with a zero exponent is the subnormal c * 2^-24 (times 2^k
//    for a field at bit k of its half), which the tensor cores multiply
//    exactly.  The MMAs of a score are grouped by k: the pairs at the same
//    bit position share an accumulator, scaled by 2^-k once per score;
//  * scores: mma.sync m16n8k16 with A = key codes (16 tokens x 16 channels)
//    and B = the folded query q_c Δ_c split exactly into hi = fp16(q Δ) and
//    lo = q Δ - hi in two columns per head, so every product is exact and the
//    fp32 accumulation is as good as an fp32 dot product; a second MMA adds
//    Σ_c q_c min_c (q·k̂_t = Σ_c (q_c Δ_c) code_tc + Σ_c q_c min_c exactly);
//  * online softmax in log2 units, rescaled only when the running max grows
//    by more than 2^8 (the stale max keeps every p <= 256);
//  * fp16 range: a query row whose largest |q_c| exceeds 1 is stored scaled
//    by 2^-e (so q_c Δ_c stays inside fp16 for every fp16 Δ_c; the scores
//    take 2^e back), the values of a unit by 2^F (so small Δ_t keep P' out of
//    the fp16 subnormals), and a chunk whose P' would pass 65504 raises the
//    head's softmax reference by a power of two; all three are exact;
//  * values: Oᵀ += Vᵀ P' with A = value codes (16 channels x 16 tokens: a
//    channel's tokens are contiguous in the block) and B = p_t Δ_t 2^-k split
//    into hi/lo fp16; P' moves from the score layout to the B layout through
//    a per-warp shared buffer whose layout keeps both sides free of bank
//    conflicts; Σ_t p_t min_t is added per head.
// Tails go through the same tensor-core path: the fp16 ring rows are A
// operands as they are (values transposed by ldmatrix), and the fp32 sink
// rows are narrowed to fp16 exactly (they were fp16 when appended).
//
// Pre-RoPE keys (the ROPE instantiations): q R(aθ) k̂ = (R(-a0 θ) q) (R(jθ) k̂)
// with a0 the first position of a group or tail chunk and j < G; the query
// rows are turned back per group, each dequantized key turned by its offset
// from a table, and both split into hi/lo fp16 operands (rope_chunk_scores).
//
// Host io (the HIO instantiations, word-rule widths): q, out and the fresh
// token's rows are pinned host memory mapped into the device; the warps load
// the query and fresh rows with plain 16-byte loads where the device
// instantiation issues bulk copies, and the merge writes the output there.
//
// Outlier tables (the OUTL instantiations; KV-cache quantization guide
// (pigeon), "KVQuant adds": a small share of values kept in fp16 beside the
// codes).  An outlier's code is 0, so the dense path above reads it as the
// min of its vector; the kernel adds the difference.  The tables travel
// with the block in the same bulk copy.  Keys: a score lane walks the
// table's rows of its own TPL tokens and adds q_c (x - min_c) scaled to log2
// units; key outliers sit in fixed channels and spread over the tokens, so
// this takes no barrier and no atomic.  Values: outliers bunch in the few
// tokens of large scale, so the lanes take the chunk's entries in turn
// (entry-parallel) and add p_h,t (x - min_t) for the four heads into a
// per-warp fp32 [4][D] buffer with shared atomics; p comes from the score
// lanes through a per-warp [4][CH] exchange.  The buffer is at the running
// max: its owner lanes (the lane that holds that output channel) rescale it
// with the accumulators and add it to their output at the close of a unit.
#pragma once

#include "kivi_internal.cuh"

#include <math.h>

#include <type_traits>

namespace kivi {
namespace mma {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;                         // lazy rescale threshold (log2 units)
constexpr unsigned long long kWaitNs = 2000000000ull;    // bounded wait: 2 s
constexpr float kTwo24 = 16777216.0f;                    // codes enter the MMAs scaled by 2^-24

// error word bits
constexpr unsigned kErrCopy = 1u;   // a copy never completed
constexpr unsigned kErrSlot = 2u;   // a combine never released the slots
constexpr unsigned kClaim = 2u;     // positions a warp claims at a time

struct Args {
  Geo g;
  const uint8_t* arena;
  const __half* q;
  __half* out;
  float* partials;      // [B * nq * h_q][stride][d + 4]: o[d], m, l, 2 pad
  unsigned* counters;   // [units]: CTAs finished per unit
  unsigned* error;      // kErrCopy | kErrSlot (debug builds also kErrIndex | kErrNonFinite)
  unsigned long long wait_ns;   // how long a warp waits for a copy before it gives up (kErrCopy)
  DecodePlan plan;
  int32_t ns;           // copy stages per warp
  int32_t stage_bytes;  // bytes per stage (block bytes rounded up to 128)
  int32_t stride;       // partial records per (sequence, query head)
  int32_t npass;        // head passes (4 query rows each) per kv head: ceil(nq * rep / 4)
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
  int fresh;       // 1 = the token being appended, fp16 rows from the inputs
  int n;           // tokens in the chunk (0 only when there is nothing to attend to)
  int first;       // first sink index, or first ring token (0-based, oldest first)
};
// Tail position idx of a unit: the sink chunks, the ring chunks, then (fused
// append) the fresh token.
__device__ __forceinline__ TailChunk tail_chunk(int idx, int n_sink, int n_res, bool fresh) {
  TailChunk t;
  const int n_sc = (n_sink + kSinkChunk - 1) / kSinkChunk;
  const int n_rc = (n_res + kRingChunk - 1) / kRingChunk;
  t.fresh = 0;
  if (idx < n_sc) {
    t.sink = 1;
    t.first = idx * kSinkChunk;
    t.n = min(kSinkChunk, n_sink - t.first);
  } else if (fresh && idx == n_sc + n_rc) {
    t.sink = 0;
    t.fresh = 1;
    t.first = 0;
    t.n = 1;
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
// The same, but a thread whose phase is not complete is suspended (issuing
// nothing) until it completes or about `hint_ns` nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for a barrier phase: one non-blocking test first (the usual case: the
// copy landed while the warp computed), then suspended rather than spinning
// (a spinning warp would take issue slots from the warps that compute); gives
// up once the wait has lasted `limit_ns` and reports false.  A limit of 1 ns
// gives up at once unless the phase is already complete (a test of the expiry
// path: the copies still arrive, and the try_wait forms may suspend the
// thread until they do).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  if (limit_ns <= 1) return false;
  const uint32_t hint = limit_ns < 1000000ull ? static_cast<uint32_t>(limit_ns) : 1000000u;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (global_ns() - t0 >= limit_ns) return false;
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two transposed 8x8 fp16 tiles: lanes 0-7 address the rows of tile 0, lanes
// 8-15 those of tile 1 (16-byte aligned); lane 4i + j receives elements
// (2j, i) and (2j + 1, i) of each tile.
__device__ __forceinline__ void ldsm_x2_trans(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}

// Shared-memory loads at 32-bit shared addresses (ordered like other memory
// operations: the stage they read is handed back to the copy engine later).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Lane-0 work without a divergent branch: PTX predicated on `pred`.
__device__ __forceinline__ uint32_t atom_add_shared_if(bool pred, uint32_t addr, uint32_t v) {
  uint32_t old = 0u;
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p atom.shared.add.u32 %0, [%1], %3;\n\t}"
               : "+r"(old) : "r"(addr), "r"(static_cast<uint32_t>(pred)), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void sts32_if(bool pred, uint32_t addr, uint32_t v) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.shared.u32 [%0], %1;\n\t}"
               :: "r"(addr), "r"(v), "r"(static_cast<uint32_t>(pred)) : "memory");
}
// Arms the barrier for `bytes` and issues one bulk copy of them, if pred.
__device__ __forceinline__ void bulk_load_if(bool pred, uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
               "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %2;\n\t"
               "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "r"(static_cast<uint32_t>(pred)) : "memory");
}

// An arrival that completes the stage's phase with no copy (a debug build's
// skipped copy whose address failed its check).
__device__ __forceinline__ void mbar_arrive_if(bool pred, uint32_t bar) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
               :: "r"(bar), "r"(static_cast<uint32_t>(pred)) : "memory");
}

// A warp copies `bytes` (a multiple of 16) from global memory into shared
// memory with plain 16-byte loads (the host-io instantiations: pinned host
// memory mapped into the device, read over the chip-to-chip link); the caller
// then completes the stage.  Out of line: it takes no registers from the loop.
static __device__ __noinline__ void warp_copy16(uint8_t* dst, const void* src, int bytes) {
  const int lane = threadIdx.x & 31;
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = lane; i < bytes / 16; i += 32) d[i] = s[i];
}
// Orders a lane's generic-proxy writes into a stage before the bulk copies
// (async proxy) that later reuse it.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// 2^x by the SFU (PTX ex2.approx, subnormal results flushed to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------- code pairs
// A lane's slice of a packed row is cut into pairs of adjacent channels
// (tokens for values): pair p = elements 2p and 2p + 1.  The packing puts
// element j of a 32-bit word in half j & 1 at bit BITS * (j >> 1), so both
// elements of a pair sit at the same bit of their halves.  Bits 8..15 are
// first moved down by 8 (a shift, or a byte permute for 8-bit codes).
template <int BITS>
__host__ __device__ constexpr int pair_kb(int p) {   // bit position after the move
  return (BITS * (p % (16 / BITS))) % 8;
}
template <int BITS>
__host__ __device__ constexpr bool pair_hi(int p) {  // codes in bits 8..15
  return BITS * (p % (16 / BITS)) >= 8;
}

// Widths packed as a bit stream (b outside {2, 4, 8}): element j of a slice
// at bit b j of its words taken as one little-endian bit string.
template <int BITS>
__host__ __device__ constexpr bool stream_bits() { return !(BITS == 2 || BITS == 4 || BITS == 8); }

// fp16x2 of pair p as exact subnormals: low half = element 2p, high half =
// element 2p + 1, each code * 2^(pair_kb(p) - 24) (bit-stream widths: both
// codes moved to bit 0 of their halves, class 0).
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* w, int p) {
  if constexpr (stream_bits<BITS>()) {
    constexpr uint32_t M = (1u << BITS) - 1u;
    const int bit = 2 * BITS * p, wi = bit >> 5, sh = bit & 31;
    const uint32_t t = (sh + 2 * BITS <= 32) ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh);
    return (t & M) | ((t << (16 - BITS)) & (M << 16));
  }
  const uint32_t x = w[p / (16 / BITS)];
  if constexpr (BITS == 8) {
    return pair_hi<BITS>(p) ? prmt(x, 0u, 0x4341u) : (x & 0x00FF00FFu);
  } else {
    const uint32_t y = pair_hi<BITS>(p) ? (x >> 8) : x;
    return y & (((1u << BITS) - 1u) * (0x00010001u << pair_kb<BITS>(p)));
  }
}

// Key pairs in the order the score MMAs take them: grouped by bit position
// (class), so that both pairs of one MMA share a class.  n indexes the sorted
// list of the NP pairs.
template <int BITS, int NP>
__host__ __device__ constexpr int ord_pair(int n) {
  if constexpr (stream_bits<BITS>()) {
    return n;
  } else if constexpr (BITS == 4) {
    const int cls = n / (NP / 2), k = n % (NP / 2);
    return 4 * (k / 2) + 2 * (k % 2) + cls;
  } else if constexpr (BITS == 2) {
    const int cls = n / (NP / 4), k = n % (NP / 4);
    return 8 * (k / 2) + 4 * (k % 2) + cls;
  } else {
    return n;
  }
}
template <int BITS>
__host__ __device__ constexpr int n_acc() { return stream_bits<BITS>() ? 1 : BITS == 2 ? 4 : 2; }
// accumulator of the score MMA that takes sorted pairs 2j, 2j + 1
template <int BITS, int NP>
__host__ __device__ constexpr int acc_of(int j) {
  if constexpr (stream_bits<BITS>()) return 0;
  return BITS == 8 ? (j & 1) : pair_kb<BITS>(ord_pair<BITS, NP>(2 * j)) / (BITS == 4 ? 4 : 2);
}
// 2^-k of accumulator a
template <int BITS>
__host__ __device__ constexpr float acc_scale(int a) {
  if constexpr (stream_bits<BITS>()) return 1.f;
  return BITS == 8 ? 1.f : BITS == 4 ? (a ? 0.0625f : 1.f) : (a == 0 ? 1.f : a == 1 ? 0.25f : a == 2 ? 0.0625f : 0.015625f);
}

__device__ __forceinline__ float warp_max_rows(float v) {   // over the 8 lanes that share lane & 3
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float warp_sum_rows(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// CTA that owns work position x when W positions are cut into P ranges
// [floor(c W / P), floor((c + 1) W / P)).
__device__ __forceinline__ int owner_of(int64_t x, int64_t W, int64_t P) {
  const int64_t c = ((x + 1) * P - 1) / W;
  return static_cast<int>(c < P - 1 ? c : P - 1);
}

// Byte offset of P'[column (head h, part e)][token t] in a warp's exchange
// buffer.  With 32-token chunks the two parts of a head share a 128-byte
// block, in opposite 64-byte halves, and the 16-byte segments are swizzled
// by head, so that the score-layout writes (4 heads x 4 token quads) and the
// B-layout reads (one column's 8 tokens per lane) both hit 32 distinct banks.
template <int CH>
__device__ __forceinline__ uint32_t xch_off(int h, int e, int t) {
  if constexpr (CH == 32) {
    return 128u * h + 64u * ((e + h) & 1) + 16u * ((t >> 3) ^ (2 * ((h >> 1) & 1))) + 2u * (t & 7);
  } else {
    return 32u * (2 * h + e) + 2u * t;
  }
}

// Shared-memory layout (byte sizes) of one warp; the host sizes the launch
// with the same formulas.
template <int D, int CH>
struct WarpSmem {
  static constexpr int kQS = D / 2 + 16;          // a quarter row of q (D/4 fp16) plus 16 bytes of padding
  static constexpr int kQRow = 4 * kQS;
  static constexpr int kQ = 4 * kQRow;            // four heads
  static constexpr int kSlot = 4 * (D + 4) * 4;   // four heads: o[D], m, l (+ 2 pad)
  static constexpr int kXch = CH == 32 ? 512 : 256;
};

// Unit u as (sequence bb, kv head hk, head pass).  A decode orders units
// pass-fastest; several query tokens (MQ) order them pass-slowest, so that
// with a grid of a multiple of npass CTAs the passes of one group block are
// processed at the same moment by CTAs npass apart (one DRAM read, the other
// passes served by L2).
template <bool MQ>
__device__ __forceinline__ void unit_parts(const Args& a, int u, int& bb, int& hk, int& pass) {
  if constexpr (MQ) {
    const int u0 = a.g.B * a.g.hkv;
    pass = u / u0;
    bb = (u % u0) / a.g.hkv;
    hk = u % a.g.hkv;
  } else {
    const int per_b = a.g.hkv * a.npass;
    bb = u / per_b;
    hk = (u % per_b) / a.npass;
    pass = u % a.npass;
  }
}

// Row (of q, out and the partial records: [B][q_rows][h_q]) of query row hh
// of unit u.  MQ: query tokens in rows q_rows apart per sequence; otherwise
// nq = q_rows = 1 and the rows of a pass are adjacent heads.
template <bool MQ>
__device__ __forceinline__ int64_t q_row(const Args& a, int u, int hh) {
  int bb, hk, pass;
  unit_parts<MQ>(a, u, bb, hk, pass);
  if constexpr (MQ) {
    const int v = 4 * pass + hh;   // row of the kv head: query token v / rep, head v % rep
    return (static_cast<int64_t>(bb) * a.plan.q_rows + v / a.g.rep) * a.g.hq + hk * a.g.rep + v % a.g.rep;
  } else {
    return static_cast<int64_t>(bb) * a.g.hq + hk * a.g.rep + 4 * pass + hh;
  }
}
// Query rows of unit u (at most four).
template <bool MQ>
__device__ __forceinline__ int unit_rows(const Args& a, int u) {
  int bb, hk, pass;
  unit_parts<MQ>(a, u, bb, hk, pass);
  return min(4, (MQ ? a.plan.nq : 1) * a.g.rep - 4 * pass);
}

// Merge of the `total` partial records (o[D], m, l, pad, pad) of one query
// head for channels ch, ch + 1: M = max m_s, w_s = 2^(m_s - M),
// L = Σ l_s w_s, O = Σ o_s w_s.  The loads of up to kMergeBatch records go
// out together (one L2 round trip per batch), one rescale per batch.
constexpr int kMergeBatch = 16;
template <int D>
__device__ __forceinline__ void merge_partials(const float* base, int total, int ch, float2& O, float& L) {
  float m = -INFINITY;
  O = make_float2(0.f, 0.f);
  L = 0.f;
  for (int s0 = 0; s0 < total; s0 += kMergeBatch) {
    float2 ml[kMergeBatch], o[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      if (s0 + k < total) {
        const float* ps = base + (s0 + k) * (D + 4);
        ml[k] = __ldcg(reinterpret_cast<const float2*>(ps + D));
        o[k] = __ldcg(reinterpret_cast<const float2*>(ps + ch));
      } else {
        ml[k] = make_float2(-INFINITY, 0.f);
        o[k] = make_float2(0.f, 0.f);
      }
    }
    float mb = m;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) mb = fmaxf(mb, ml[k].x);
    if (mb == -INFINITY) continue;
    const float sc = (m == -INFINITY) ? 0.f : ex2(m - mb);
    O.x *= sc;
    O.y *= sc;
    L *= sc;
    m = mb;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const float f = (ml[k].x == -INFINITY) ? 0.f : ex2(ml[k].x - m);
      O.x = fmaf(o[k].x, f, O.x);
      O.y = fmaf(o[k].y, f, O.y);
      L = fmaf(ml[k].y, f, L);
    }
  }
}

// Merges channel pair i (query row i / (D/2)) of unit u and writes it out.
template <int D, bool MQ>
__device__ __forceinline__ void merge_out(const Args& a, int u, int i, int total) {
  const int hh = i / (D / 2), ch = 2 * (i % (D / 2));
  const int64_t row = q_row<MQ>(a, u, hh);
  float2 O;
  float L;
  merge_partials<D>(a.partials + row * a.stride * (D + 4), total, ch, O, L);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<__half2*>(a.out + row * D + ch) = __floats2half2_rn(O.x * inv, O.y * inv);
}

// Combines head hh of the nw warp slots (o[D], m, l, pad, pad) for channel ch.
template <int D>
__device__ __forceinline__ void combine_slots(const float* slots, int slot_floats, int nw, int hh, int ch,
                                              float& M, float& L, float& O) {
  M = -INFINITY;
  for (int w = 0; w < nw; ++w) M = fmaxf(M, slots[w * slot_floats + hh * (D + 4) + D]);
  L = 0.f;
  O = 0.f;
  if (M == -INFINITY) return;
  for (int w = 0; w < nw; ++w) {
    const float* so = slots + w * slot_floats + hh * (D + 4);
    const float mw = so[D];
    const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
    L = fmaf(so[D + 1], f, L);
    O = fmaf(so[ch], f, O);
  }
}

// A combined (M, L, O) of channel ch of query head `head`: the output when
// the unit lies inside one CTA, else this CTA's partial record.
template <int D>
__device__ __forceinline__ void publish(const Args& a, int64_t head, int ch, int total, int cslot, float M,
                                        float L, float O) {
  if (total == 1) {
    a.out[head * D + ch] = __float2half_rn(L > 0.f ? O / L : 0.f);
  } else {
    if (kDebugChecks && (cslot < 0 || cslot >= a.stride)) {   // a record outside the head's stride
      atomicOr(a.error, kErrIndex);
      return;
    }
    float* dst = a.partials + (head * a.stride + cslot) * (D + 4);
    dst[ch] = O;
    if (ch == 0) { dst[D] = M; dst[D + 1] = L; }
  }
}

// Epilogue of a unit that is not the CTA's last, run by the last warp to sign
// in: combines the slots, publishes, releases the slots (s_done) and, in the
// unit's last CTA, merges the partials.
template <int D, bool MQ>
__device__ __forceinline__ void warp_epilogue(const Args& a, const float* slots, int slot_floats, int nw, int u,
                                           int nh, int total, int cslot, int useq, unsigned* s_done) {
  const int lane = threadIdx.x & 31;
  for (int hh = 0; hh < nh; ++hh) {
    const int64_t row = q_row<MQ>(a, u, hh);
    // per head: the max and the slot weights once, channels lane + 32 j
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, slots[w * slot_floats + hh * (D + 4) + D]);
    float L = 0.f, O[D / 32];
#pragma unroll
    for (int j = 0; j < D / 32; ++j) O[j] = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < nw; ++w) {
        const float* so = slots + w * slot_floats + hh * (D + 4);
        const float mw = so[D];
        const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        L = fmaf(so[D + 1], f, L);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) O[j] = fmaf(so[lane + 32 * j], f, O[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < D / 32; ++j) publish<D>(a, row, lane + 32 * j, total, cslot, M, L, O[j]);
  }
  __syncwarp();
  __threadfence_block();
  if (lane == 0) *reinterpret_cast<volatile unsigned*>(s_done) = static_cast<unsigned>(useq + 1);
  if (total == 1) return;
  __threadfence();
  __syncwarp();
  unsigned last_cta = 0;
  if (lane == 0) last_cta = (atomicAdd(a.counters + u, 1u) == static_cast<unsigned>(total - 1)) ? 1u : 0u;
  last_cta = __shfl_sync(0xffffffffu, last_cta, 0);
  if (!last_cta) return;
  __threadfence();
  for (int i = lane; i < nh * D / 2; i += 32) merge_out<D, MQ>(a, u, i, total);
  if (lane == 0) a.counters[u] = 0u;
}

// Epilogue of the CTA's last unit, run by every thread of the CTA.
// `others_done`: every other CTA of the unit had published its record when a
// warp of this CTA read the unit's counter (with acquire order), so this CTA
// is the unit's last: it merges as soon as its own record is written, without
// the release fence and the sign-in (the counter, at total - 1, is reset for
// the next launch).  Otherwise it publishes, signs in, and the CTA that signs
// in last merges.
template <int D, bool MQ>
__device__ __forceinline__ void cta_epilogue(const Args& a, const float* slots, int slot_floats, int nw, int u,
                                          int nh, int total, int cslot, unsigned* s_flag, bool others_done) {
  for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
    const int hh = i / D, ch = i % D;
    float M, L, O;
    combine_slots<D>(slots, slot_floats, nw, hh, ch, M, L, O);
    publish<D>(a, q_row<MQ>(a, u, hh), ch, total, cslot, M, L, O);
  }
  if (total == 1) return;
  if (others_done) {
    __syncthreads();   // this CTA's record is visible to all of its threads
  } else {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_flag = (atomicAdd(a.counters + u, 1u) == static_cast<unsigned>(total - 1)) ? 1u : 0u;
    __syncthreads();
    if (!*s_flag) return;
    __threadfence();
  }
  for (int i = threadIdx.x; i < nh * D / 2; i += blockDim.x) merge_out<D, MQ>(a, u, i, total);
  if (threadIdx.x == 0) a.counters[u] = 0u;
}

// Scores of one chunk (CH tokens) for the lane's head c: lane (r, c) gets
// the tokens TPL r + i of the chunk, rowa / rowb the shared addresses of its
// first key-row pair (odd r of 64-byte rows swapped: sw).  bq holds the folded
// query of the lane's B column, scs the scale of the accumulated codes, cst_h
// the head's Σ q_c min_c.
// Words of a lane's key quarter: whole words, except a bit-stream quarter
// of 2 b bytes at head dim 64 for odd b (it may start on a 16-bit boundary:
// one word more, shifted down by ksh bits).
template <int D, int BITS>
__host__ __device__ constexpr bool key_quarter_unaligned() { return stream_bits<BITS>() && (D * BITS / 32) % 4 != 0; }
template <int D, int BITS>
__host__ __device__ constexpr int key_quarter_words() {
  return key_quarter_unaligned<D, BITS>() ? (D * BITS / 32 + 2 + 3) / 4 : (D * BITS / 8) / 16;
}

template <int D, int BITS, int CH>
__device__ __forceinline__ void chunk_scores(const uint32_t (&bq)[D / 8], uint32_t rowa, uint32_t rowb, float scs,
                                             float cst_h, int sw, int ksh, float (&sv)[CH / 8]) {
  constexpr int RK = D * BITS / 8, KW = key_quarter_words<D, BITS>(), NP = D / 8, NKC = D / 16, TPL = CH / 8;
  constexpr int NA = n_acc<BITS>();
#pragma unroll
  for (int v2 = 0; v2 < TPL / 2; ++v2) {
    uint32_t w0[KW], w1[KW];
    const uint32_t row0 = rowa + 2 * v2 * RK;
    const uint32_t row1 = rowb + 2 * v2 * RK;
    if constexpr (key_quarter_unaligned<D, BITS>()) {   // from the 4-byte boundary below, shifted down
#pragma unroll
      for (int i = 0; i < KW; ++i) {
        w0[i] = lds32(row0 + 4 * i);
        w1[i] = lds32(row1 + 4 * i);
      }
#pragma unroll
      for (int i = 0; i < KW; ++i) {
        w0[i] = i + 1 < KW ? __funnelshift_r(w0[i], w0[i + 1], ksh) : (w0[i] >> ksh);
        w1[i] = i + 1 < KW ? __funnelshift_r(w1[i], w1[i + 1], ksh) : (w1[i] >> ksh);
      }
    } else if constexpr (stream_bits<BITS>()) {   // a quarter of b words, 4-byte aligned
#pragma unroll
      for (int i = 0; i < KW; ++i) {
        w0[i] = lds32(row0 + 4 * i);
        w1[i] = lds32(row1 + 4 * i);
      }
    } else if constexpr (KW >= 4) {
#pragma unroll
      for (int i = 0; i < KW; i += 4) {
        const uint4 x = lds128(row0 + 4 * i);
        const uint4 y = lds128(row1 + 4 * i);
        w0[i] = x.x; w0[i + 1] = x.y; w0[i + 2] = x.z; w0[i + 3] = x.w;
        w1[i] = y.x; w1[i + 1] = y.y; w1[i + 2] = y.z; w1[i + 3] = y.w;
      }
    } else if constexpr (KW == 2) {
      const uint2 x = lds64(row0);
      const uint2 y = lds64(row1);
      w0[0] = x.x; w0[1] = x.y; w1[0] = y.x; w1[1] = y.y;
    } else {
      w0[0] = lds32(row0);
      w1[0] = lds32(row1);
    }
    float acc[NA][4];
#pragma unroll
    for (int i = 0; i < NA; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int j = 0; j < NKC; ++j) {
      const int pa = ord_pair<BITS, NP>(2 * j), pb = ord_pair<BITS, NP>(2 * j + 1);
      mma16816(acc[acc_of<BITS, NP>(j)], code_pair<BITS>(w0, pa), code_pair<BITS>(w1, pa),
               code_pair<BITS>(w0, pb), code_pair<BITS>(w1, pb), bq[pa], bq[pb]);
    }
    float s_a = (acc[0][0] + acc[0][1]) * acc_scale<BITS>(0);
    float s_b = (acc[0][2] + acc[0][3]) * acc_scale<BITS>(0);
#pragma unroll
    for (int i = 1; i < NA; ++i) {
      s_a = fmaf(acc[i][0] + acc[i][1], acc_scale<BITS>(i), s_a);
      s_b = fmaf(acc[i][2] + acc[i][3], acc_scale<BITS>(i), s_b);
    }
    s_a = fmaf(s_a, scs, cst_h);
    s_b = fmaf(s_b, scs, cst_h);
    sv[2 * v2] = sw ? s_b : s_a;
    sv[2 * v2 + 1] = sw ? s_a : s_b;
  }
}

// ---------------------------------------------------------- pre-RoPE keys
// Keys stored before the rotary embedding (KV-cache quantization guide
// (pigeon), "KVQuant adds").  The score of the key at position a is
// q · R(a θ) k̂_a.  With a = a0 + j (a0 the first position of a frozen group
// or a tail chunk, j < G), R(a θ) = R(a0 θ) R(j θ) and R is orthogonal, so
//   q · R(a θ) k̂ = (R(-a0 θ) q) · (R(j θ) k̂):
// the query rows are turned back by the base angle once per group (the B
// operand, split into hi/lo fp16 halves as the folded query of the plain
// decode), and each dequantized key is turned by its offset's angle, taken
// from a fixed table (rope.cu), in fp32 and split into hi/lo fp16 A
// operands, so both factors of every product are exact to 22 bits.  The score
// k-chunk kc pairs each channel with its rotation partner: k = 2c + e is
// channel RS c + 2 kc + e of the first half and k = 8 + 2c + e the same channel
// of the second half (RS = D/8), so lane (r, c) holds both channels of each
// pair it turns and reads two contiguous RS-channel regions of a key row.
//
// cos and sin of a θ by the Cody-Waite reduction (W. J. Cody and W. Waite,
// "Software Manual for the Elementary Functions", 1980): θ is carried as
// th_hi + th_lo, a th_hi is split exactly into p + e with one fma, the
// multiple k of 2π nearest to a θ is taken off p with 2π in two fp32 parts
// (k times the first part is exact in the fma), then the small terms are
// added.  Positions from 2^24 on, which fp32 does not hold exactly, reduce in
// double.
constexpr float kInv2Pi = 0.15915494309189535f;
constexpr float kTwoPiHi = 6.28318548202514648f;      // fl(2π)
constexpr float kTwoPiLo = -1.7484555314695172e-7f;   // 2π - fl(2π)
__device__ __forceinline__ float2 h2f(uint32_t x) { return __half22float2(*reinterpret_cast<const __half2*>(&x)); }

__device__ __forceinline__ float2 rope_cs(int64_t a, float th_hi, float th_lo) {
  float r;
  if (a < (int64_t{1} << 24)) {
    const float af = static_cast<float>(a);
    const float p = af * th_hi;
    const float e = fmaf(af, th_hi, -p);
    const float t = fmaf(af, th_lo, e);
    const float k = rintf((p + t) * kInv2Pi);
    r = fmaf(-k, kTwoPiHi, p);
    r = fmaf(-k, kTwoPiLo, r) + t;
  } else {
    const double x = static_cast<double>(a) * (static_cast<double>(th_hi) + static_cast<double>(th_lo));
    r = static_cast<float>(x - 6.283185307179586476925 * rint(x * 0.15915494309189533576888));
  }
  float sn, cs;
  __sincosf(r, &sn, &cs);
  return make_float2(cs, sn);
}

template <int D>
struct Rope {
  static constexpr int kRS = D / 8;                  // channels of a lane's region per half
  static constexpr int kRowBytes = (D / 2 + 8) * 8;  // a warp's angle row: (cos, sin) per pair, regions 16 B apart
  static constexpr int kQRow = 2 * D + 4;            // query rows in natural order, 4 bytes of padding
  __host__ __device__ static constexpr int idx(int i) { return i + 2 * (i / kRS); }
};

// The warp's angle row for base position a: (cos, sin)(a θ_i), i < D/2.
// tab: the RoPE tables ([θ hi, lo] per pair first).
template <int D>
__device__ __forceinline__ void rope_angles(float2* wrow, const float* __restrict__ tab, int64_t a) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = lane; i < D / 2; i += 32) {
    const float2 th = __ldg(reinterpret_cast<const float2*>(tab) + i);
    wrow[Rope<D>::idx(i)] = rope_cs(a, th.x, th.y);
  }
  __syncwarp();
}

// fp16 pair of x0, x1: their high parts (11 significant bits, exact in fp16)
// or the rest
__device__ __forceinline__ uint32_t rope_split(float x0, float x1, bool lo) {
  const float h0 = __uint_as_float(__float_as_uint(x0) & 0xFFFFE000u);
  const float h1 = __uint_as_float(__float_as_uint(x1) & 0xFFFFE000u);
  return lo ? pack_half2(x0 - h0, x1 - h1) : pack_half2(h0, h1);
}

// B fragment pair of R(-a0 θ) q for the lane's column and k-chunk kc (made
// when needed rather than kept live): query row at qrow_s (natural order),
// part lo (odd column) or hi; the warp's angle row at wrow_s.
template <int D>
__device__ __forceinline__ void rope_fold_kc(uint32_t& b0, uint32_t& b1, int kc, uint32_t qrow_s, uint32_t wrow_s,
                                             int c, bool lo) {
  constexpr int RS = Rope<D>::kRS, H = D / 2;
  const int i = RS * c + 2 * kc;
  const float2 qa = h2f(lds32(qrow_s + 2 * i));
  const float2 qb = h2f(lds32(qrow_s + 2 * (i + H)));
  const uint4 w = lds128(wrow_s + 8 * Rope<D>::idx(i));   // (cos, sin) of pairs i and i + 1
  const float c0 = __uint_as_float(w.x), s0 = __uint_as_float(w.y);
  const float c1 = __uint_as_float(w.z), s1 = __uint_as_float(w.w);
  // R(-φ) (x, y) = (c x + s y, c y - s x)
  b0 = rope_split(fmaf(c0, qa.x, s0 * qb.x), fmaf(c1, qa.y, s1 * qb.y), lo);
  b1 = rope_split(fmaf(c0, qb.x, -s0 * qa.x), fmaf(c1, qb.y, -s1 * qa.y), lo);
}

// Codes of a lane's key region: NW words from the 4-byte boundary at or below
// its first code, shifted so that the region starts at bit 0.  Word rule: a
// region is whole words, except 16 channels of 2 bits (head dim 64), whose
// codes sit in bits 8..15 of both halves of their word for odd c; bit streams:
// RS b bits from bit RS c b.
template <int D, int BITS>
struct RopeCodes {
  static constexpr int RS = Rope<D>::kRS;
  static constexpr bool kStream = stream_bits<BITS>();
  static constexpr int NW = kStream ? (RS * BITS + 24 + 31) / 32 : (RS * BITS >= 32 ? RS * BITS / 32 : 1);
  static constexpr int kHalfBytes = (D / 2) * BITS / 8;   // the second half's region is this far on
  // byte offset of the region's first word and the shift inside it, for c
  __device__ static void where(int c, uint32_t& off, int& sh) {
    const int bit = RS * c * BITS;
    off = static_cast<uint32_t>(bit >> 5) * 4u;
    sh = kStream ? (bit & 31) : ((bit & 31) >> 1);
  }
  __device__ static void load(uint32_t (&w)[NW], uint32_t addr, int sh) {
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = lds32(addr + 4 * i);
    if constexpr (kStream) {
#pragma unroll
      for (int i = 0; i < NW; ++i) w[i] = i + 1 < NW ? __funnelshift_r(w[i], w[i + 1], sh) : (w[i] >> sh);
    } else if constexpr (RS * BITS < 32) {
      w[0] >>= sh;   // bits crossing from the high half into the low one are masked off below
    }
  }
  // the two codes of local pair k (channels RS c + 2k, + 1) in the low and
  // high halves of one word, each at bit pair_shift(k) of its half: the fp16
  // subnormals code 2^(pair_shift(k) - 24), which convert to fp32 exactly
  __device__ static constexpr int pair_shift(int k) {
    return kStream ? 0 : (BITS * (k % (16 / BITS)) + BITS <= 10 ? BITS * (k % (16 / BITS))
                                                                  : BITS * (k % (16 / BITS)) - 8);
  }
  template <int N>
  __device__ static uint32_t pair_h(const uint32_t (&w)[N], int k) {
    constexpr uint32_t M = (1u << BITS) - 1u;
    if constexpr (kStream) {
      const int bit = 2 * BITS * k, wi = bit >> 5, s = bit & 31;
      const uint32_t t = (s + 2 * BITS <= 32 || wi + 1 >= N) ? (w[wi] >> s) : __funnelshift_r(w[wi], w[wi + 1], s);
      return (t & M) | ((t << (16 - BITS)) & (M << 16));
    } else {
      constexpr int PPW = 16 / BITS;
      const int s = BITS * (k % PPW);
      const uint32_t x = w[k / PPW];
      return s + BITS <= 10 ? x & ((M * 0x00010001u) << s) : (x >> 8) & ((M * 0x00010001u) << (s - 8));
    }
  }
  // the two codes of local pair k (channels RS c + 2k, + 1) as floats
  __device__ static void pair(const uint32_t (&w)[NW], int k, float& f0, float& f1) {
    constexpr uint32_t M = (1u << BITS) - 1u;
    uint32_t lo, hi;
    if constexpr (kStream) {
      const int bit = 2 * BITS * k, wi = bit >> 5, s = bit & 31;
      const uint32_t t = (s + 2 * BITS <= 32 || wi + 1 >= NW) ? (w[wi] >> s) : __funnelshift_r(w[wi], w[wi + 1], s);
      lo = t & M;
      hi = (t >> BITS) & M;
    } else {
      constexpr int PPW = 16 / BITS;   // pairs per word
      const uint32_t x = (w[k / PPW] >> (BITS * (k % PPW))) & (M * 0x00010001u);
      lo = x & 0xFFFFu;
      hi = x >> 16;
    }
    // 2^23 + code, then 2^23 off: exact
    f0 = __uint_as_float(0x4B000000u | lo) - 8388608.f;
    f1 = __uint_as_float(0x4B000000u | hi) - 8388608.f;
  }
};

// Scores of a frozen group's chunk (CH tokens from s0) for pre-RoPE keys:
// lane (r, c) gets head c's scores of tokens s0 + TPL r + i, the same layout as
// chunk_scores.  kq, ks: shared addresses of the block's key codes and key
// (Δ, min) rows; otab: the offset table; scs: the score scale.
template <int D, int BITS, int CH>
__device__ __forceinline__ void rope_chunk_scores(uint32_t qrow_s, uint32_t wrow_s, uint32_t kq, uint32_t ks, int s0,
                                                  int sw, const float4* __restrict__ otab, int G, float scs,
                                                  float (&sv)[CH / 8]) {
  using RC = RopeCodes<D, BITS>;
  constexpr int RS = Rope<D>::kRS, H = D / 2, TPL = CH / 8, NT = TPL / 2, RK = D * BITS / 8, NW = RC::NW;
  const int lane = threadIdx.x & 31, r = lane >> 2, c = lane & 3;
  uint32_t roff;
  int rsh;
  RC::where(c, roff, rsh);
  // the code regions of the lane's tokens: tile v2, token e (A row r or r + 8),
  // half.  Bit streams load a region's words up front; the word rule loads
  // each word when its first pair comes up (fewer live registers)
  constexpr int PPW = RC::kStream ? 1 : 16 / BITS;   // pairs per word (word rule)
  uint32_t w[NT][2][2][RC::kStream ? NW : 1];
  uint32_t rows[NT][2];
#pragma unroll
  for (int v2 = 0; v2 < NT; ++v2) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      rows[v2][e] = kq + static_cast<uint32_t>((s0 + TPL * r + 2 * v2 + (e ^ sw)) * RK) + roff;
      if constexpr (RC::kStream) {
        RC::load(w[v2][e][0], rows[v2][e], rsh);
        RC::load(w[v2][e][1], rows[v2][e] + RC::kHalfBytes, rsh);
      }
    }
  }
  float acc[NT][4];
#pragma unroll
  for (int v2 = 0; v2 < NT; ++v2) acc[v2][0] = acc[v2][1] = acc[v2][2] = acc[v2][3] = 0.f;
#pragma unroll
  for (int kc = 0; kc < D / 16; ++kc) {
    const int i = RS * c + 2 * kc;
    uint32_t b0, b1;
    rope_fold_kc<D>(b0, b1, kc, qrow_s, wrow_s, c, (r & 1) != 0);
    // Δ scaled by 2^(24 - pair_shift): the codes arrive as fp16 subnormals
    const float sk = __uint_as_float(static_cast<uint32_t>(127 + 24 - RC::pair_shift(kc)) << 23);
    float2 da = h2f(lds32(ks + 2 * i));
    float2 db = h2f(lds32(ks + 2 * (i + H)));
    da.x *= sk; da.y *= sk; db.x *= sk; db.y *= sk;
    const float2 ma = h2f(lds32(ks + 2 * D + 2 * i));
    const float2 mb = h2f(lds32(ks + 2 * D + 2 * (i + H)));
    if constexpr (!RC::kStream) {
      if (kc % PPW == 0) {   // the words holding pairs kc .. kc + PPW - 1
#pragma unroll
        for (int v2 = 0; v2 < NT; ++v2) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t x0 = lds32(rows[v2][e] + 4 * (kc / PPW));
            uint32_t x1 = lds32(rows[v2][e] + RC::kHalfBytes + 4 * (kc / PPW));
            if constexpr (RS * BITS < 32) { x0 >>= rsh; x1 >>= rsh; }
            w[v2][e][0][0] = x0;
            w[v2][e][1][0] = x1;
          }
        }
      }
    }
#pragma unroll
    for (int v2 = 0; v2 < NT; ++v2) {
      uint32_t ah[4], al[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = s0 + TPL * r + 2 * v2 + (e ^ sw);   // the token's offset in its group
        const int kk = RC::kStream ? kc : kc % PPW;        // the pair within the loaded word(s)
        const float2 xc = h2f(RC::pair_h(w[v2][e][0], kk)), yc = h2f(RC::pair_h(w[v2][e][1], kk));
        const float x0 = fmaf(xc.x, da.x, ma.x), x1 = fmaf(xc.y, da.y, ma.y);
        const float y0 = fmaf(yc.x, db.x, mb.x), y1 = fmaf(yc.y, db.y, mb.y);
        const float4 rr = __ldg(otab + (i / 2) * (G + 1) + j);   // (cos, sin) / 2 of pairs i and i + 1
        const float2 r0 = make_float2(rr.x, rr.y), r1 = make_float2(rr.z, rr.w);
        // R(φ) (x, y) = (c x - s y, s x + c y), halved by the table
        const float u0 = fmaf(r0.x, x0, -r0.y * y0), v0 = fmaf(r0.y, x0, r0.x * y0);
        const float u1 = fmaf(r1.x, x1, -r1.y * y1), v1 = fmaf(r1.y, x1, r1.x * y1);
        ah[e] = rope_split(u0, u1, false);
        al[e] = rope_split(u0, u1, true);
        ah[2 + e] = rope_split(v0, v1, false);
        al[2 + e] = rope_split(v0, v1, true);
      }
      mma16816(acc[v2], ah[0], ah[1], ah[2], ah[3], b0, b1);
      mma16816(acc[v2], al[0], al[1], al[2], al[3], b0, b1);
    }
  }
#pragma unroll
  for (int v2 = 0; v2 < NT; ++v2) {
    const float s_a = (acc[v2][0] + acc[v2][1]) * scs, s_b = (acc[v2][2] + acc[v2][3]) * scs;
    sv[2 * v2] = sw ? s_b : s_a;
    sv[2 * v2 + 1] = sw ? s_a : s_b;
  }
}

template <bool RG>
using RunTableT = typename std::conditional<RG, RunTable, NoRuns>::type;

// The kernel body.  RG: a ragged launch; per-unit plan values come from the
// run table `rt` (the unit's run) instead of the launch's plan.  ROPE: keys
// stored before the rotary embedding, turned at their positions in the score
// products (see rope_chunk_scores).
template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL, bool ROPE, bool HIO>
__device__ __forceinline__ void decode_body(const Args& a, const RunTableT<RG>& rt) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  using WS = WarpSmem<D, CH>;
  // outlier corrections (OUTL): per warp a [4][CH] fp32 exchange of the
  // chunk's p and the [4][D] fp32 value corrections
  constexpr int kCorr = OUTL ? 16 * (CH + D) : 0;
  // pre-RoPE keys: per warp the angle row of the current group or tail chunk
  constexpr int kRopeRow = ROPE ? Rope<D>::kRowBytes : 0;
  static_assert(!(ROPE && OUTL), "pre-RoPE keys take no outlier tables");
  constexpr int RK = D * BITS / 8;          // key row bytes
  constexpr int KW = RK / 16;               // 32-bit words of a lane's key quarter
  constexpr int QD = D / 4;                 // channels of a lane's quarter
  constexpr int NP = QD / 2;                // channel pairs of a lane's quarter
  constexpr int NKC = D / 16;               // k-chunks over channels
  constexpr int QV = CH * BITS / 4;         // bits of a lane's value quarter per chunk of CH tokens
  constexpr int VW = QV >= 32 ? QV / 32 : 1;
  constexpr int TPL = CH / 8;               // tokens per score lane per chunk
  constexpr int NCT = D / 16;               // channel tiles
  constexpr int NKT = CH / 16;              // token k-chunks per chunk (value MMA)
  constexpr int NA = n_acc<BITS>();

  const Geo& g = a.g;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int rep = g.rep;
  const float qscale = kLog2e * rsqrtf(static_cast<float>(D));
  const int64_t n_vis = a.plan.n_vis_groups;
  const int64_t P = gridDim.x;
  int64_t W;
  if constexpr (RG) W = rt.W; else W = static_cast<int64_t>(a.units) * a.uw;
  const int64_t c_start = (static_cast<int64_t>(blockIdx.x) * W) / P;
  const int64_t c_end = (static_cast<int64_t>(blockIdx.x + 1) * W) / P;
  if (c_start >= c_end) return;   // uniform; only when W < P, which the host avoids
  // ragged launches: the run holding work position x, the run of unit u
  // (searched upwards from a run k at or before it), a unit's first position
  auto run_at = [&](int64_t x) -> int {
    int k = 0;
    if constexpr (RG) while (k + 1 < rt.n && rt.r[k + 1].pos0 <= x) ++k;
    return k;
  };
  auto run_of = [&](int u, int k) -> int {
    if constexpr (RG) while (k + 1 < rt.n && u >= rt.r[k + 1].ubase) ++k;
    return k;
  };
  auto unit_start = [&](int u, int k) -> int64_t {
    if constexpr (RG) return rt.r[k].pos0 + static_cast<int64_t>(u - rt.r[k].ubase) * rt.r[k].uw;
    else return static_cast<int64_t>(u) * a.uw;
  };
  auto unit_width = [&](int k) -> int {
    if constexpr (RG) return rt.r[k].uw;
    else return static_cast<int>(a.uw);
  };
  int k_first = 0, k_last = 0;
  int u_first, u_last;
  if constexpr (RG) {
    k_first = run_at(c_start);
    k_last = run_at(c_end - 1);
    u_first = rt.r[k_first].ubase + static_cast<int>((c_start - rt.r[k_first].pos0) / rt.r[k_first].uw);
    u_last = rt.r[k_last].ubase + static_cast<int>((c_end - 1 - rt.r[k_last].pos0) / rt.r[k_last].uw);
  } else {
    u_first = static_cast<int>(c_start / a.uw);
    u_last = static_cast<int>((c_end - 1) / a.uw);
  }

  // shared memory: stages | q | slots | exchange | barriers | item rings (per warp, warp-major within each)
  uint8_t* stages = smem_raw;
  uint8_t* q_all = stages + static_cast<size_t>(nw) * a.ns * a.stage_bytes;
  float* slots = reinterpret_cast<float*>(q_all + nw * WS::kQ);
  uint8_t* xch_all = reinterpret_cast<uint8_t*>(slots) + nw * WS::kSlot;
  float* corr_all = reinterpret_cast<float*>(xch_all + nw * WS::kXch);
  uint8_t* rope_all = reinterpret_cast<uint8_t*>(corr_all) + nw * kCorr;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rope_all + nw * kRopeRow);
  __shared__ unsigned s_arrive;   // warps signed in for the current combine
  __shared__ unsigned s_done;     // combines completed
  __shared__ unsigned s_flag;     // this CTA merges its last unit
  __shared__ unsigned s_next;     // positions of the CTA's range claimed so far
  __shared__ float s_qf[kDecodeWarps][4];    // per warp: the query prescale 2^e of each row of the open unit
  __shared__ float s_vsc[kDecodeWarps][2];   // per warp: the open unit's value scale 2^F (0: not chosen), 2^-F

  uint8_t* my_stages = stages + static_cast<size_t>(warp) * a.ns * a.stage_bytes;
  uint8_t* qw = q_all + warp * WS::kQ;
  uint8_t* xw = xch_all + warp * WS::kXch;
  float* pbuf = corr_all + warp * (kCorr / 4);   // [4][CH]: p of (head, token) of the open chunk
  float* ocorr = pbuf + 4 * CH;                  // [4][D], real scale, at the running max
  const uint32_t xw_s = smem_addr(xw);
  float2* wrow = reinterpret_cast<float2*>(rope_all + warp * kRopeRow);   // pre-RoPE keys: the angle row
  // pre-RoPE keys: the rotation tables in the arena's workspace (θ, then the
  // offsets' (cos, sin) / 2), read through the read-only cache
  const float* rtab = ROPE ? reinterpret_cast<const float*>(a.arena + g.ws_rope) : nullptr;
  const uint32_t bar0 = smem_addr(bars + warp * a.ns);
  int* ring_w = reinterpret_cast<int*>(bars + nw * a.ns) + warp * a.ns;   // this warp's item ring
  const uint32_t blk_bytes = static_cast<uint32_t>(g.block_bytes);

  // a launch that follows in the stream may start its own set-up now; it
  // waits below for this grid to finish before it reads or writes memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) { s_arrive = 0u; s_done = 0u; s_next = 0u; s_flag = 0u; }
  if (lane == 0) {
    for (int s = 0; s < a.ns; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // the previous kernel in the stream (an append, or the last step's decode)
  // has completed and its writes are visible from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");

  auto unit_base = [&](int u) -> const uint8_t* {
    int bb, hk, pass;
    unit_parts<MQ>(a, u, bb, hk, pass);
    return a.arena + (static_cast<int64_t>(bb) * g.hkv + hk) * g.unit_bytes;
  };
  // (sequence, kv head) index of unit u
  auto unit_kv = [&](int u) -> int64_t {
    int bb, hk, pass;
    unit_parts<MQ>(a, u, bb, hk, pass);
    return static_cast<int64_t>(bb) * g.hkv + hk;
  };

  // ------------------------------------------------------------ producer
  // per-warp copy pipeline.  Lane 0 claims the CTA's positions kClaim at a
  // time from a shared counter (so a warp that is held up takes fewer), and before
  // the first position of a unit it issues that unit's query rows; each item
  // is noted in the warp's ring (one int per stage: 2 * rel for a position
  // rel of the CTA's range, 2 * k + 1 for the query rows of unit u_first + k)
  const uint32_t n_slots = static_cast<uint32_t>(g.n_slots);
  const bool ring_slots = g.window > 0;
  const int t_sink = static_cast<int>(a.plan.st.n_sink), t_res = static_cast<int>(a.plan.st.n_res);
  const bool fresh = a.plan.k_fresh != nullptr;   // fused append: the fresh token closes every tail
  const int rs0 = static_cast<int>((a.plan.st.n_groups * g.G) % g.R);   // ring slot of the oldest ring token
  const int range = static_cast<int>(c_end - c_start);
  // slot of the first visible group (ring of slots with a window); a unit's
  // visible groups never outnumber its slots
  const uint32_t slot0 = ring_slots ? static_cast<uint32_t>(a.plan.g_first % g.n_slots)
                                    : static_cast<uint32_t>(a.plan.g_first);
  // per-unit plan values: the launch's (uniform) or the unit's run's (ragged)
  auto f_nvis = [&](int k) -> int {
    if constexpr (RG) return rt.r[k].n_vis; else return static_cast<int>(n_vis);
  };
  auto f_slot0 = [&](int k) -> uint32_t {
    if constexpr (RG) return rt.r[k].slot0; else return slot0;
  };
  auto f_sink = [&](int k) -> int {
    if constexpr (RG) return rt.r[k].n_sink; else return t_sink;
  };
  auto f_res = [&](int k) -> int {
    if constexpr (RG) return rt.r[k].n_res; else return t_res;
  };
  auto f_rs0 = [&](int k) -> int {
    if constexpr (RG) return rt.r[k].rs0; else return rs0;
  };
  auto f_gfirst = [&](int k) -> int64_t {
    if constexpr (RG) return rt.r[k].g_first; else return a.plan.g_first;
  };
  auto f_qpos0 = [&](int k) -> int64_t {
    if constexpr (RG) return rt.r[k].q_pos0; else return a.plan.q_pos0;
  };
  auto f_fresh_pos = [&](int k) -> int64_t {
    if constexpr (RG) return rt.r[k].fresh_pos; else return a.plan.fresh_pos;
  };
  int c_st = 0;                 // consumer: stage, phase parity
  uint32_t c_ph = 0;
  int inflight = 0;             // items issued and not yet consumed (warp-uniform)
  int p_st = 0;                 // producer: next stage
  int p_u = -1;                 // unit (from u_first) of the last claimed position
  bool p_have = false;          // a claimed position waits for a stage
  bool p_q = false;             // the query rows of unit p_u wait for a stage
  bool p_done = false;          // the CTA's positions are all claimed (and the last claim used up)
  int p_rel = 0;
  int p_next = 0, p_left = 0;   // the warp's current claim: next position, positions left in it
  // end of unit p_u's positions, relative to c_start (negative or zero before the first claim)
  int p_end = static_cast<int>(unit_start(u_first, k_first) - c_start);
  int p_k = k_first;            // run of unit p_u (ragged launches)
  const uint8_t* p_unit = nullptr;
  bool aborted = false;
  const uint32_t stages_s = smem_addr(my_stages);
  const uint32_t ring_s = smem_addr(ring_w);
  const uint32_t next_s = smem_addr(&s_next);
  const bool leader = lane == 0;
  // the whole warp runs the bookkeeping on warp-uniform values; lane 0 alone
  // claims, notes the item and issues the copies (predicated, no branch)
  auto produce = [&]() {
    if (aborted) return;
    while (inflight < a.ns) {
      if (!p_have) {
        if (p_left == 0) {   // claim the next kClaim positions of the range
          if (p_done) return;
          // kClaim positions at a time while the range is far from done, one
          // at a time over its last 2 nw positions (the CTA's warps then
          // finish closer together); the leader reads the counter plainly
          // to choose, so the choice may be a claim late, which is harmless
          int packed = 0;
          if (leader) {
            const unsigned seen = *reinterpret_cast<volatile unsigned*>(&s_next);
            const unsigned k = seen + 2u * static_cast<unsigned>(nw) < static_cast<unsigned>(range) ? kClaim : 1u;
            packed = static_cast<int>(2u * atom_add_shared_if(true, next_s, k) + (k - 1u));
          }
          packed = __shfl_sync(0xffffffffu, packed, 0);
          const int rel = packed >> 1;
          if (rel >= range) { p_done = true; return; }
          p_next = rel;
          p_left = min((packed & 1) + 1, range - rel);
        }
        p_rel = p_next++;
        --p_left;
        p_have = true;
        if (p_rel >= p_end) {   // the position lies in a later unit (positions only grow)
          do {
            ++p_u;
            p_k = run_of(u_first + p_u, p_k);
            p_end += unit_width(p_k);
          } while (p_rel >= p_end);
          p_unit = unit_base(u_first + p_u);
          p_q = true;
        }
      }
      const uint32_t dst = stages_s + p_st * a.stage_bytes;
      const uint32_t bar = bar0 + 8 * p_st;
      if (p_q) {
        const int uq = u_first + p_u;
        const int nh_q = unit_rows<MQ>(a, uq);
        sts32_if(leader, ring_s + 4 * p_st, 2 * p_u + 1);
        if constexpr (HIO) {   // the rows from host memory, loaded by the warp
          uint8_t* dsts = my_stages + static_cast<size_t>(p_st) * a.stage_bytes;
          for (int hh = 0; hh < nh_q; ++hh) warp_copy16(dsts + hh * D * 2, a.q + q_row<MQ>(a, uq, hh) * D, 2 * D);
          fence_proxy_async();
          __syncwarp();
          mbar_arrive_if(leader, bar);
        } else if constexpr (MQ) {
          if (lane == 0) {   // one copy per query row (the rows of a pass need not be adjacent)
            bulk_arm(bar, static_cast<uint32_t>(nh_q) * D * 2);
            for (int hh = 0; hh < nh_q; ++hh)
              bulk_copy(dst + hh * D * 2, a.q + q_row<MQ>(a, uq, hh) * D, 2 * D, bar);
          }
        } else {             // adjacent heads: one copy
          bulk_load_if(leader, dst, a.q + q_row<MQ>(a, uq, 0) * D, static_cast<uint32_t>(nh_q) * D * 2, bar);
        }
        p_q = false;
        if (++p_st == a.ns) p_st = 0;
        ++inflight;
        continue;
      }
      const int pos = p_rel - (p_end - unit_width(p_k));   // position inside unit p_u
      bool issued = true;
      const int p_nvis = f_nvis(p_k);
      if (pos < p_nvis) {   // a frozen group block
        uint32_t slot = f_slot0(p_k) + static_cast<uint32_t>(pos);
        if (ring_slots && slot >= n_slots) slot -= n_slots;
        sts32_if(leader, ring_s + 4 * p_st, 2 * p_rel);
        const uint8_t* src = p_unit + g.groups + static_cast<int64_t>(slot) * g.block_bytes;
        if (dbg_in_region(g, src, blk_bytes)) bulk_load_if(leader, dst, src, blk_bytes, bar);
        else mbar_arrive_if(leader, bar);
      } else {                // a tail chunk: key rows then value rows
        const TailChunk tk = tail_chunk(pos - p_nvis, f_sink(p_k), f_res(p_k), fresh);
        if (tk.n == 0) {
          issued = false;     // nothing to copy or to attend to
        } else if (HIO && tk.fresh) {   // the appended token's rows from host memory
          const int64_t row = unit_kv(u_first + p_u) * D;
          uint8_t* dsts = my_stages + static_cast<size_t>(p_st) * a.stage_bytes;
          warp_copy16(dsts, a.plan.k_fresh + row, 2 * D);
          warp_copy16(dsts + 16 * D, a.plan.v_fresh + row, 2 * D);
          sts32_if(leader, ring_s + 4 * p_st, 2 * p_rel);
          fence_proxy_async();
          __syncwarp();
          mbar_arrive_if(leader, bar);
        } else if (lane == 0) {
          ring_w[p_st] = 2 * p_rel;
          if (tk.fresh) {     // the appended token's rows, straight from the inputs
            const int64_t row = unit_kv(u_first + p_u) * D;
            bulk_arm(bar, 4 * D);
            bulk_copy(dst, a.plan.k_fresh + row, 2 * D, bar);
            bulk_copy(dst + 16 * D, a.plan.v_fresh + row, 2 * D, bar);
          } else if (tk.sink) {
            const uint32_t bytes = static_cast<uint32_t>(tk.n) * D * 4;
            const uint8_t* sk = p_unit + g.sink_k + static_cast<int64_t>(tk.first) * D * 4;
            const uint8_t* sv = p_unit + g.sink_v + static_cast<int64_t>(tk.first) * D * 4;
            if (dbg_in_region(g, sk, bytes) && dbg_in_region(g, sv, bytes)) {
              bulk_arm(bar, 2 * bytes);
              bulk_copy(dst, sk, bytes, bar);
              bulk_copy(dst + 16 * D, sv, bytes, bar);
            } else {
              mbar_arrive_if(true, bar);
            }
          } else {
            int s0 = f_rs0(p_k) + tk.first;
            if (s0 >= g.R) s0 -= g.R;
            const int n1 = min(tk.n, g.R - s0), n2 = tk.n - n1;   // the ring may wrap
            const uint8_t* rk = p_unit + g.res_k + static_cast<int64_t>(s0) * D * 2;
            const uint8_t* rv = p_unit + g.res_v + static_cast<int64_t>(s0) * D * 2;
            if (dbg_in_region(g, rk, n1 * D * 2) && dbg_in_region(g, rv, n1 * D * 2) &&
                dbg_in_region(g, p_unit + g.res_k, n2 * D * 2) && dbg_in_region(g, p_unit + g.res_v, n2 * D * 2)) {
              bulk_arm(bar, static_cast<uint32_t>(tk.n) * D * 4);
              bulk_copy(dst, rk, n1 * D * 2, bar);
              bulk_copy(dst + 16 * D, rv, n1 * D * 2, bar);
              if (n2 > 0) {
                bulk_copy(dst + n1 * D * 2, p_unit + g.res_k, n2 * D * 2, bar);
                bulk_copy(dst + 16 * D + n1 * D * 2, p_unit + g.res_v, n2 * D * 2, bar);
              }
            } else {
              mbar_arrive_if(true, bar);
            }
          }
        }
      }
      p_have = false;
      if (issued) {
        if (++p_st == a.ns) p_st = 0;
        ++inflight;
      }
    }
  };
  // waits for the consumer's current stage; false after an abort
  auto acquire = [&]() -> bool {
    if (aborted) return false;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * c_st, c_ph, a.wait_ns));   // warp-uniform verdict
    if (!ok) {
      aborted = true;
      if (lane == 0) atomicOr(a.error, kErrCopy);
    }
    return ok;
  };
  auto release = [&]() {
    __syncwarp();
    if (++c_st == a.ns) { c_st = 0; c_ph ^= 1u; }
    --inflight;
  };

  // this lane's B column r = (head r >> 1, part r & 1), channel quarter c
  const uint32_t partmask = (r & 1) ? 0xFFFFFFFFu : 0u;
  const int hh_col = r >> 1;
  // P' of score-layout token TPL*r + i enters value pair ((TPL*r + i) % (CH/4)) / 2,
  // whose codes sit at bit k: p is scaled by 2^-k in fp32 before the hi/lo split
  auto vscl_at = [&](int i) -> float {
    const int l = (TPL * r + i) % (CH / 4);
    const int kb = stream_bits<BITS>() ? 0 : (BITS * ((l / 2) % (16 / (stream_bits<BITS>() ? 1 : BITS)))) % 8;
    return __uint_as_float(static_cast<uint32_t>(127 - kb) << 23);
  };
  float vscl[TPL];
#pragma unroll
  for (int i = 0; i < TPL; ++i) vscl[i] = vscl_at(i);
  const float sc_scale = qscale * kTwo24;

  // per-lane shared-memory offsets inside a group block (loop invariant)
  constexpr bool kSwap = (RK == 64);   // 64-byte key rows: odd r swaps its row pair
  const int sw = kSwap ? (r & 1) : 0;
  // a lane's quarter of a key row starts at byte c RK/4; at head dim 64 a
  // bit-stream quarter (2 b bytes) may start on a 16-bit boundary: its words
  // are read from the 4-byte boundary below and shifted down by ksh bits
  const uint32_t q_off = static_cast<uint32_t>(c * (RK / 4));
  const int ksh = static_cast<int>(8 * (q_off & 3u));
  const uint32_t o_k0 = static_cast<uint32_t>(g.blk_kq) + (TPL * r + sw) * RK + (q_off & ~3u);
  const uint32_t o_k1 = static_cast<uint32_t>(g.blk_kq) + (TPL * r + 1 - sw) * RK + (q_off & ~3u);
  const uint32_t o_ds = static_cast<uint32_t>(g.blk_ks) + c * (D / 2);   // key Δ; key min at + 2D
  const uint32_t o_vs = static_cast<uint32_t>(g.blk_vs) + TPL * r * 4;   // value (Δ, min) of token TPL*r
  const uint32_t vrow = static_cast<uint32_t>(g.G) * BITS / 8;           // bytes of one value-code row
  const uint32_t vrow8 = 8 * vrow, vrow16 = 16 * vrow;
  // bit streams: the lane's 8 codes of a 32-token chunk start at bit 8 c b
  // of the chunk; the word holding that bit and the shift inside it
  constexpr bool kStream = stream_bits<BITS>();
  const uint32_t o_vq = kStream ? static_cast<uint32_t>(g.blk_vq) + r * vrow + 4 * ((8 * c * BITS) >> 5)
                                : static_cast<uint32_t>(g.blk_vq) + r * vrow +
                                      (QV >= 32 ? c * (QV / 8) : ((c * QV) / 32) * 4);
  const int vsh = kStream ? (8 * c * BITS) & 31
                          : (QV >= 32 ? 0 : ((c * QV) % 32) / 2);   // the lane's codes within their word

  // ------------------------------------------------------------ consumer
  const int nunits = u_last - u_first + 1;
  int cu = -1;                  // open unit (from u_first); -1 before the first
  int nh = 0, total = 1, cslot = 0;
  int u_rel = 0;                // first position of the open unit, relative to c_start
  float res_m = -INFINITY, res_l = 0.f, res_mn = 0.f;
  bool o_real = false;          // oacc holds real-scale values (after a tail chunk)
  float oacc[NCT][4];
#pragma unroll
  for (int i = 0; i < NCT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const uint8_t* qlane = qw + hh_col * WS::kQRow + c * WS::kQS;
  const uint32_t q_s = smem_addr(qlane);
  // q of row hh, channel ch from the q area (16-byte chunks of 4 pairs, stored
  // in pair order 0, 2, 1, 3; quarters padded)
  auto q_at = [&](int hh, int ch) -> float {
    const int idx = ch >> 3, w = (ch >> 1) & 3;
    const int slot = (w == 1) ? 2 : (w == 2) ? 1 : w;
    const __half* p = reinterpret_cast<const __half*>(qw + hh * WS::kQRow + (idx / (QD / 8)) * WS::kQS +
                                                      (idx % (QD / 8)) * 16 + slot * 4);
    return __half2float(p[ch & 1]);
  };

  // the prescale 2^e of query row c (this lane's score head) of the open unit
  auto head_qf = [&]() -> float { return s_qf[threadIdx.x >> 5][threadIdx.x & 3]; };
  // P' = p Δ_t 2^(F - k): a power of two 2^F per unit, chosen from the largest
  // Δ_t of the warp's first frozen chunk of the unit, keeps the fp16 pair of
  // P' away from the subnormals when the values are small (the rounding of a
  // subnormal hi half is not caught by the lo half); the accumulators give
  // 2^-F back when they turn to real scale.  In the warp's s_vsc: 2^F (0 until chosen), then 2^-F
  auto value_unscale = [&]() -> float {
    const float* v = s_vsc[threadIdx.x >> 5];
    return v[0] == 0.f ? 1.f : v[1];
  };

  // token masks, needed with a window or with several query tokens: this
  // lane's score column c is query row 4 pass + c of the open unit, i.e.
  // query token jq at position hi = q_pos0 + jq, which sees the positions
  // [lo, hi] with lo = hi + 1 - W (a window) and every sink up to hi.  With
  // one query token (jq = 0, hi = T - 1) only a window masks anything, and
  // only in frozen groups (the ring and the sinks lie inside any window)
  int jq = 0;
  int c_k = k_first;            // run of the open unit (ragged launches)
  auto masked = [&]() { return MQ || g.window > 0; };
  auto col_hi = [&]() -> int64_t { return f_qpos0(c_k) + (MQ ? jq : 0); };
  auto col_lo = [&](int64_t hi) { return g.window > 0 ? hi + 1 - g.window : static_cast<int64_t>(INT64_MIN); };
  auto open_unit = [&](int k) {
    const int u = u_first + k;
    nh = unit_rows<MQ>(a, u);
    if constexpr (MQ) jq = (4 * (u / (g.B * g.hkv)) + c) / rep;   // pass-slowest order
    c_k = run_of(u, c_k);
    const int64_t u_base = unit_start(u, c_k);
    u_rel = static_cast<int>(u_base - c_start);
    const int first = owner_of(u_base, W, P);
    total = owner_of(u_base + unit_width(c_k) - 1, W, P) - first + 1;
    cslot = static_cast<int>(blockIdx.x) - first;
    res_m = -INFINITY; res_l = 0.f; res_mn = 0.f;
    o_real = false;
    if (lane == 0) s_vsc[warp][0] = 0.f;   // the unit's value scale: not chosen yet
#pragma unroll
    for (int i = 0; i < NCT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    if constexpr (OUTL) {   // this lane's entries: head c, channels 16 ct + r (+ 8)
#pragma unroll
      for (int ct = 0; ct < NCT; ++ct) { ocorr[c * D + 16 * ct + r] = 0.f; ocorr[c * D + 16 * ct + r + 8] = 0.f; }
    }
  };
  auto rescale_corr = [&](float corr) {
    if constexpr (OUTL) {
#pragma unroll
      for (int ct = 0; ct < NCT; ++ct) { ocorr[c * D + 16 * ct + r] *= corr; ocorr[c * D + 16 * ct + r + 8] *= corr; }
    }
  };
  // the warp's state of unit cu into its slot, then the sign-in: the last warp
  // combines a unit that is not the CTA's last while the others stream on; the
  // CTA's last unit is combined by every thread once all streaming is over
  auto close_unit = [&]() {
    const int u = u_first + cu;
    float lh = warp_sum_rows(res_l), mh = warp_sum_rows(res_mn);
    // the slot may be rewritten once the combine of the previous unit is done
    if (lane == 0) {
      const volatile unsigned* done = &s_done;
      if (*done < static_cast<unsigned>(cu)) {
        const unsigned long long t0 = global_ns();
        while (*done < static_cast<unsigned>(cu)) {
          __nanosleep(64);
          if (global_ns() - t0 > kWaitNs) { atomicOr(a.error, kErrSlot); break; }
        }
      }
    }
    __syncwarp();
    __threadfence_block();
    float* my_slot = slots + warp * (WS::kSlot / 4);
    if (c < nh) {
      float* so = my_slot + c * (D + 4);
      if (r == 0) { so[D] = res_m; so[D + 1] = lh; }
      const float osc = o_real ? 1.f : kTwo24 * value_unscale();
#pragma unroll
      for (int ct = 0; ct < NCT; ++ct) {
        so[16 * ct + r] = fmaf(oacc[ct][0] + oacc[ct][1], osc, mh);
        so[16 * ct + r + 8] = fmaf(oacc[ct][2] + oacc[ct][3], osc, mh);
        if constexpr (OUTL) {
          so[16 * ct + r] += ocorr[c * D + 16 * ct + r];
          so[16 * ct + r + 8] += ocorr[c * D + 16 * ct + r + 8];
        }
      }
    }
    if (cu != nunits - 1) {
      __threadfence_block();
      __syncwarp();
      unsigned last = 0;
      if (lane == 0) last = (atomicAdd(&s_arrive, 1u) == static_cast<unsigned>(nw - 1)) ? 1u : 0u;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence_block();
        if (lane == 0) s_arrive = 0u;
        warp_epilogue<D, MQ>(a, slots, WS::kSlot / 4, nw, u, nh, total, cslot, cu, &s_done);
      }
    } else {
      // the CTA's last unit: each warp looks at the unit's counter as it
      // arrives (the other CTAs' parts usually ended long before), so the
      // load's latency hides behind the wait for the slowest warp
      if (lane == 0 && total > 1 && ld_acquire_gpu(a.counters + u) == static_cast<unsigned>(total - 1))
        atomicOr(&s_flag, 1u);
      __syncthreads();
      cta_epilogue<D, MQ>(a, slots, WS::kSlot / 4, nw, u, nh, total, cslot, &s_flag, s_flag != 0u);
    }
  };

  for (;;) {
    produce();
    __syncwarp();
    if (inflight == 0) break;   // every claim issued and consumed
    if (!acquire()) break;
    const int item = static_cast<int>(lds32(ring_s + 4 * c_st));
    if (item & 1) {
      // ------------------------------------------------------ query rows
      // of the next unit this warp works on; units passed on the way are closed
      const int k = item >> 1;
      while (cu < k) {
        if (cu >= 0) close_unit();
        ++cu;
        open_unit(cu);
      }
      // copied to this warp's q area: quarter rows padded by 16 bytes, heads
      // past nh zero.  A row whose largest |q_c| exceeds 1 is stored scaled by
      // 2^-e (exact: a power of two) so that its largest |q_c| is below 1;
      // the folded q_c Δ_c is then at most Δ_c, inside the fp16 range for
      // every fp16 Δ_c, and the scores take 2^e back (head_qf, kept in the
      // row's first quarter padding).
      const uint8_t* src = my_stages + c_st * a.stage_bytes;
#pragma unroll
      for (int kk = lane; kk < 4 * D / 8; kk += 32) {
        const int hh = kk / (D / 8), idx = kk % (D / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (hh < nh) v = *reinterpret_cast<const uint4*>(src + hh * D * 2 + idx * 16);
        // the largest |q_c| of the row as fp16 bits (magnitudes order as
        // their bit patterns), then its exponent
        uint32_t mb = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        mb = max(mb & 0xFFFFu, mb >> 16);
#pragma unroll
        for (int o = 1; o < D / 8; o <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));   // the row's chunks
        // m in [2^(e-1), 2^e) for m > 1: m 2^-e below 1
        const int e = mb > 0x3C00u ? static_cast<int>(mb >> 10) - 14 : 0;
        if constexpr (kDebugChecks) {
          if (mb >= 0x7C00u) atomicOr(a.error, kErrNonFinite);   // an inf or NaN query element
        }
        if (e > 0) {
          // 2^-e as an fp16 pair (e <= 16: a normal number or a subnormal)
          const uint32_t h = e <= 14 ? static_cast<uint32_t>(15 - e) << 10 : 1u << (24 - e);
          const uint32_t s2 = h | (h << 16);
          v.x = hmul2_u(v.x, s2); v.y = hmul2_u(v.y, s2); v.z = hmul2_u(v.z, s2); v.w = hmul2_u(v.w, s2);
        }
        if constexpr (ROPE) {
          // natural channel order, rows 2D + 4 bytes apart (a lane's reads of
          // its two regions then fall on distinct banks)
          uint32_t* dq = reinterpret_cast<uint32_t*>(qw + hh * Rope<D>::kQRow + idx * 16);
          dq[0] = v.x; dq[1] = v.y; dq[2] = v.z; dq[3] = v.w;
        } else {
          // pairs (0, 1, 2, 3) of the chunk stored as (0, 2, 1, 3): the Σ q·min
          // MMAs then take their B pairs straight from one 16-byte load
          *reinterpret_cast<uint4*>(qw + hh * WS::kQRow + (idx / (QD / 8)) * WS::kQS + (idx % (QD / 8)) * 16) =
              make_uint4(v.x, v.z, v.y, v.w);
        }
        if (idx == 0) s_qf[warp][hh] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
      }
      release();
      __syncwarp();
      continue;
    }
    const int pos = (item >> 1) - u_rel;   // position inside the open unit
    const int c_nvis = f_nvis(c_k);
    if (pos < c_nvis) {
      // ------------------------------------------------------ a frozen group
      const int64_t grp = f_gfirst(c_k) + pos;
      const uint32_t blk = stages_s + c_st * a.stage_bytes;   // shared address of the block

      const float qf = head_qf();   // head c's query prescale 2^e
      const int64_t a_grp = g.S + grp * g.G;
      uint32_t bq[ROPE ? 1 : NP];
      float cst_h = 0.f, scs;
      if constexpr (ROPE) {
        // the query turned back by the group's base angle a_grp θ (hi/lo
        // columns); the keys' offsets are turned in rope_chunk_scores
        rope_angles<D>(wrow, rtab, a_grp);
        scs = 2.f * qscale * qf;   // the table halves the turned keys
      } else {
      // (1) the query (natural pair order) and the folded B fragments:
      // hi = fp16(q Δ) in even columns, lo = q Δ - hi in odd ones
      uint32_t q2[NP];   // natural pair order (the q area holds pairs 0, 2, 1, 3 of each 4)
#pragma unroll
      for (int i = 0; i < NP / 4; ++i) {
        const uint4 v = lds128(q_s + 16 * i);
        q2[4 * i] = v.x; q2[4 * i + 1] = v.z; q2[4 * i + 2] = v.y; q2[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < NP / 4; ++i) {
        const uint4 dv = lds128(blk + o_ds + 16 * i);
        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t hi = hmul2_u(q2[4 * i + j], dw[j]);
          bq[4 * i + j] = hfma2_u(q2[4 * i + j], dw[j], (hi ^ 0x80008000u) & partmask);
        }
      }
      // (2) Σ_c q_c min_c for every head (column 2c = head c).  A holds min pairs
      // 4i, 4i+1, 4i+2, 4i+3 as loaded (rows r | r+8 x k-halves); the first MMA
      // pairs row r with q of pairs 4i, 4i+2, the second row r+8 with q of
      // pairs 4i+1, 4i+3, and the two useful rows are added
      float cst_a[4] = {0.f, 0.f, 0.f, 0.f}, cst_b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < NP / 4; ++i) {
        const uint4 mv = lds128(blk + o_ds + 2 * D + 16 * i);
        mma16816(cst_a, mv.x, mv.y, mv.z, mv.w, q2[4 * i], q2[4 * i + 2]);
        mma16816(cst_b, mv.x, mv.y, mv.z, mv.w, q2[4 * i + 1], q2[4 * i + 3]);
      }
      cst_h = (cst_a[0] + cst_b[2]) * (qscale * qf);
      scs = sc_scale * qf;
      }

      for (int s0 = 0; s0 < g.G; s0 += CH) {
        // (3) scores: lane (r, c) gets head c's scores of tokens s0 + TPL*r + i
        float sv[TPL];
        if constexpr (ROPE) {
          rope_chunk_scores<D, BITS, CH>(smem_addr(qw + hh_col * Rope<D>::kQRow), smem_addr(wrow),
                                         blk + static_cast<uint32_t>(g.blk_kq), blk + static_cast<uint32_t>(g.blk_ks),
                                         s0, sw, reinterpret_cast<const float4*>(rtab + D), g.G, scs, sv);
        } else {
          const uint32_t rowa = blk + o_k0 + s0 * RK, rowb = blk + o_k1 + s0 * RK;
          chunk_scores<D, BITS, CH>(bq, rowa, rowb, scs, cst_h, sw, ksh, sv);
        }
        if constexpr (OUTL) {
          // key outliers of the lane's tokens (rows s0 + TPL r .. of the
          // table): score += q_c (x - min_c) for an entry (t, c, x), whose
          // dense part dequantized to min_c (code 0).  Key outliers sit in
          // fixed channels, so they spread over the tokens and the lanes;
          // this takes no barrier and no atomic
          const uint8_t* stg = my_stages + c_st * a.stage_bytes;
          const uint16_t* kp = reinterpret_cast<const uint16_t*>(stg + g.blk_ko);
          const uint32_t* ke = reinterpret_cast<const uint32_t*>(stg + g.blk_ko + g.out_ent);
          const __half* kmin = reinterpret_cast<const __half*>(stg + g.blk_ks) + D;
          const int t_lo = s0 + TPL * r;
          const int e1 = kp[t_lo + TPL];
          for (int e = kp[t_lo]; e < e1; ++e) {
            const uint32_t ent = ke[e];
            const int i = static_cast<int>(ent & 0xFFu) - t_lo;
            const int ch = static_cast<int>((ent >> 8) & 0xFFu);
            const float ds = (__half2float(__ushort_as_half(static_cast<unsigned short>(ent >> 16))) -
                              __half2float(kmin[ch])) * (qscale * qf * q_at(c, ch));
#pragma unroll
            for (int j = 0; j < TPL; ++j) sv[j] += (j == i) ? ds : 0.f;
          }
        }
        if (masked()) {   // tokens outside [lo, hi] are invisible to column c
          const int64_t hi = col_hi(), lo = col_lo(hi);
#pragma unroll
          for (int i = 0; i < TPL; ++i) {
            const int64_t t = a_grp + s0 + TPL * r + i;
            if (t < lo || (MQ && t > hi)) sv[i] = -INFINITY;
          }
        }
        // (4) online softmax for head c, lazy rescale: the head maxima are
        // reduced only when some lane's score exceeds its head's running max
        // by more than 2^8 (a warp vote; rare after a unit's first group)
        float mx = sv[0];
#pragma unroll
        for (int i = 1; i < TPL; ++i) mx = fmaxf(mx, sv[i]);
        if (__any_sync(0xffffffffu, mx > res_m + kRescale)) {
          mx = warp_max_rows(mx);
          if (mx > res_m + kRescale) {   // uniform over the 8 lanes of head c
            const float corr = (res_m == -INFINITY) ? 0.f : ex2(res_m - mx);
            res_m = mx;
            res_l *= corr;
            res_mn *= corr;
#pragma unroll
            for (int i = 0; i < NCT; ++i) { oacc[i][0] *= corr; oacc[i][1] *= corr; oacc[i][2] *= corr; oacc[i][3] *= corr; }
            rescale_corr(corr);
          }
        }
        const float mref = (res_m == -INFINITY) ? 0.f : res_m;   // every score so far -inf: p = 0
        float pd[TPL];
        {
          float dm[2 * TPL];   // (Δ, min) of the lane's tokens
          if constexpr (TPL == 4) {
            const uint4 x = lds128(blk + o_vs + 4 * s0);
            const uint32_t xw4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xw4[i]));
              dm[2 * i] = f.x; dm[2 * i + 1] = f.y;
            }
          } else {
            const uint2 x = lds64(blk + o_vs + 4 * s0);
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
            dm[0] = f0.x; dm[1] = f0.y; dm[2] = f1.x; dm[3] = f1.y;
          }
          // the unit's value scale 2^F, chosen by the warp's first frozen
          // chunk of the unit from its largest Δ_t
          float fsc = s_vsc[warp][0];
          if (fsc == 0.f) {
            float dmx = dm[0];
#pragma unroll
            for (int i = 1; i < TPL; ++i) dmx = fmaxf(dmx, dm[2 * i]);
            dmx = warp_max_rows(dmx);   // the chunk's largest Δ_t (the same in every lane)
            int ex = 0;
            frexpf(dmx, &ex);
            const int F = ex < 6 ? 6 - ex : 0;   // Δ_t 2^F below 2^6: p up to 2^8 keeps P' below 2^14
            fsc = __uint_as_float(static_cast<uint32_t>(127 + F) << 23);
            if (lane == 0) {
              s_vsc[warp][0] = fsc;
              s_vsc[warp][1] = __uint_as_float(static_cast<uint32_t>(127 - F) << 23);
            }
          }
#pragma unroll
          for (int i = 0; i < TPL; ++i) dm[2 * i] *= fsc;
#pragma unroll
          for (int i = 0; i < TPL; ++i) {
            const float p = ex2(sv[i] - mref);
            res_l += p;
            res_mn = fmaf(p, dm[2 * i + 1], res_mn);
            pd[i] = p * dm[2 * i] * vscl[i];
            if constexpr (OUTL) pbuf[c * CH + TPL * r + i] = p;
          }
        }
        // fp16 range of P': p_t Δ_t 2^-k (p up to 2^8 behind a lazy max) goes
        // past 65504 only for values spanning more than about 2^8 (2^b - 1)
        // within one token.  One vote per chunk; then head c's reference is
        // raised by a power of two E (res_m + E in log2 units), which scales
        // p, l, Σ p min, the accumulators and P' by 2^-E exactly, so P' stays
        // below 2^15 and nothing else changes
        {
          float pm = pd[0];
#pragma unroll
          for (int i = 1; i < TPL; ++i) pm = fmaxf(pm, pd[i]);
          if (__any_sync(0xffffffffu, pm > 65504.f)) {
            pm = warp_max_rows(pm);   // head c's largest P' of the chunk
            int ex = 0;
            frexpf(pm, &ex);
            const int E = pm > 65504.f ? ex - 15 : 0;   // pm 2^-E in [2^14, 2^15)
            if (E > 0) {
              const float corr = __uint_as_float(static_cast<uint32_t>(127 - E) << 23);
              res_m += static_cast<float>(E);
              res_l *= corr;
              res_mn *= corr;
#pragma unroll
              for (int i = 0; i < NCT; ++i) { oacc[i][0] *= corr; oacc[i][1] *= corr; oacc[i][2] *= corr; oacc[i][3] *= corr; }
              rescale_corr(corr);
#pragma unroll
              for (int i = 0; i < TPL; ++i) {
                pd[i] *= corr;
                if constexpr (OUTL) pbuf[c * CH + TPL * r + i] *= corr;
              }
            }
          }
        }
        // (5) P' hi/lo into the exchange buffer (head c, tokens TPL*r ..)
        {
          uint32_t hw[TPL / 2], lw[TPL / 2];
#pragma unroll
          for (int i = 0; i < TPL / 2; ++i) {
            const float a0 = pd[2 * i], a1 = pd[2 * i + 1];
            const float h0f = __uint_as_float(__float_as_uint(a0) & 0xFFFFE000u);
            const float h1f = __uint_as_float(__float_as_uint(a1) & 0xFFFFE000u);
            hw[i] = pack_half2(h0f, h1f);
            lw[i] = pack_half2(a0 - h0f, a1 - h1f);
          }
          if constexpr (TPL == 4) {
            *reinterpret_cast<uint2*>(xw + xch_off<CH>(c, 0, 4 * r)) = make_uint2(hw[0], hw[1]);
            *reinterpret_cast<uint2*>(xw + xch_off<CH>(c, 1, 4 * r)) = make_uint2(lw[0], lw[1]);
          } else {
            *reinterpret_cast<uint32_t*>(xw + xch_off<CH>(c, 0, 2 * r)) = hw[0];
            *reinterpret_cast<uint32_t*>(xw + xch_off<CH>(c, 1, 2 * r)) = lw[0];
          }
        }
        __syncwarp();
        if constexpr (OUTL) {
          // value outliers of the chunk, spread over the lanes by entry (they
          // bunch in the few tokens of large scale): o_h += p_h,t (x - min_t)
          // for an entry (t, c, x), whose dense part dequantized to the
          // token's min.  The owners rescaled their entries and wrote p
          // before the barrier above.
          const uint8_t* stg = my_stages + c_st * a.stage_bytes;
          const uint16_t* vp = reinterpret_cast<const uint16_t*>(stg + g.blk_vo);
          const uint32_t* ve = reinterpret_cast<const uint32_t*>(stg + g.blk_vo + g.out_ent);
          const __half* vdm = reinterpret_cast<const __half*>(stg + g.blk_vs);
          const int e1 = vp[s0 + CH];
          for (int e = vp[s0] + lane; e < e1; e += 32) {
            const uint32_t ent = ve[e];
            const int t = static_cast<int>(ent & 0xFFu);
            const int ch = static_cast<int>((ent >> 8) & 0xFFu);
            const float dx = __half2float(__ushort_as_half(static_cast<unsigned short>(ent >> 16))) -
                             __half2float(vdm[2 * t + 1]);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) atomicAdd(&ocorr[hh * D + ch], pbuf[hh * CH + t - s0] * dx);
          }
        }
        // (6) Oᵀ += Vᵀ P': B = P' of tokens c*CH/4 + 4kcn + {0,1 | 2,3} in column r
        uint32_t bp[NKT][2];
        if constexpr (NKT == 2) {
          const uint4 x = *reinterpret_cast<const uint4*>(xw + xch_off<CH>(hh_col, r & 1, 8 * c));
          bp[0][0] = x.x; bp[0][1] = x.y; bp[1][0] = x.z; bp[1][1] = x.w;
        } else {
          const uint2 x = *reinterpret_cast<const uint2*>(xw + xch_off<CH>(hh_col, r & 1, 4 * c));
          bp[0][0] = x.x; bp[0][1] = x.y;
        }
        const uint32_t vq = blk + o_vq + s0 * BITS / 8;
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct) {
          uint32_t v0[kStream ? 2 : VW], v1[kStream ? 2 : VW];
          const uint32_t rowa = vq + ct * vrow16;
          const uint32_t rowb = rowa + vrow8;
          if constexpr (kStream) {   // the lane's 8 codes: a 64-bit window from three words
            const uint32_t a0 = lds32(rowa), a1 = lds32(rowa + 4), a2 = lds32(rowa + 8);
            const uint32_t b0 = lds32(rowb), b1 = lds32(rowb + 4), b2 = lds32(rowb + 8);
            v0[0] = __funnelshift_r(a0, a1, vsh); v0[1] = __funnelshift_r(a1, a2, vsh);
            v1[0] = __funnelshift_r(b0, b1, vsh); v1[1] = __funnelshift_r(b1, b2, vsh);
          } else if constexpr (VW == 2) {
            const uint2 x = lds64(rowa), y = lds64(rowb);
            v0[0] = x.x; v0[1] = x.y; v1[0] = y.x; v1[1] = y.y;
          } else if constexpr (QV >= 32) {
            v0[0] = lds32(rowa);
            v1[0] = lds32(rowb);
          } else {
            v0[0] = lds32(rowa) >> vsh;
            v1[0] = lds32(rowb) >> vsh;
          }
#pragma unroll
          for (int kcn = 0; kcn < NKT; ++kcn) {
            mma16816(oacc[ct], code_pair<BITS>(v0, 2 * kcn), code_pair<BITS>(v1, 2 * kcn),
                     code_pair<BITS>(v0, 2 * kcn + 1), code_pair<BITS>(v1, 2 * kcn + 1), bp[kcn][0], bp[kcn][1]);
          }
        }
        __syncwarp();
      }
      release();
    } else {
      // ------------------------------------------------------ a tail chunk
      const TailChunk tk = tail_chunk(pos - c_nvis, f_sink(c_k), f_res(c_k), fresh);
      const uint8_t* kst = my_stages + c_st * a.stage_bytes;
      const uint8_t* vst = kst + 16 * D;
      if (!o_real) {   // from here on oacc holds real-scale values
        const float to_real = kTwo24 * value_unscale();
#pragma unroll
        for (int i = 0; i < NCT; ++i) { oacc[i][0] *= to_real; oacc[i][1] *= to_real; oacc[i][2] *= to_real; oacc[i][3] *= to_real; }
        o_real = true;
      }
      float s;
      if constexpr (ROPE) {
        // the chunk's tokens sit at positions a_b + r: the query turned back
        // by a_b θ, each key turned by its offset r
        const int64_t a_b = tk.fresh ? f_fresh_pos(c_k)
                          : tk.sink  ? static_cast<int64_t>(tk.first)
                                     : g.S + (f_gfirst(c_k) + f_nvis(c_k)) * g.G + tk.first;
        rope_angles<D>(wrow, rtab, a_b);
        const uint32_t qrow_s = smem_addr(qw + hh_col * Rope<D>::kQRow), wrow_s = smem_addr(wrow);
        const float4* otab = reinterpret_cast<const float4*>(rtab + D);
        constexpr int RS = Rope<D>::kRS, H = D / 2;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kc = 0; kc < NKC; ++kc) {
          const int i = RS * c + 2 * kc;
          uint32_t ah0 = 0u, ah2 = 0u, al0 = 0u, al2 = 0u;
          if (r < tk.n) {
            float2 xa, xb;   // channels (i, i + 1) and (i + H, i + H + 1) of token r
            if (tk.sink) {
              xa = *reinterpret_cast<const float2*>(kst + (r * D + i) * 4);
              xb = *reinterpret_cast<const float2*>(kst + (r * D + i + H) * 4);
            } else {
              xa = h2f(*reinterpret_cast<const uint32_t*>(kst + (r * D + i) * 2));
              xb = h2f(*reinterpret_cast<const uint32_t*>(kst + (r * D + i + H) * 2));
            }
            const float4 rr = __ldg(otab + (i / 2) * (g.G + 1) + r);
            const float2 r0 = make_float2(rr.x, rr.y), r1 = make_float2(rr.z, rr.w);
            const float u0 = fmaf(r0.x, xa.x, -r0.y * xb.x), v0 = fmaf(r0.y, xa.x, r0.x * xb.x);
            const float u1 = fmaf(r1.x, xa.y, -r1.y * xb.y), v1 = fmaf(r1.y, xa.y, r1.x * xb.y);
            ah0 = rope_split(u0, u1, false); al0 = rope_split(u0, u1, true);
            ah2 = rope_split(v0, v1, false); al2 = rope_split(v0, v1, true);
          }
          uint32_t b0, b1;
          rope_fold_kc<D>(b0, b1, kc, qrow_s, wrow_s, c, (r & 1) != 0);
          mma16816(acc, ah0, 0u, ah2, 0u, b0, b1);
          mma16816(acc, al0, 0u, al2, 0u, b0, b1);
        }
        s = (r < tk.n) ? (acc[0] + acc[1]) * (2.f * qscale * head_qf()) : -INFINITY;
      } else {
        uint32_t q2[NP];   // natural pair order
#pragma unroll
        for (int i = 0; i < NP / 4; ++i) {
          const uint4 v = lds128(q_s + 16 * i);
          q2[4 * i] = v.x; q2[4 * i + 1] = v.z; q2[4 * i + 2] = v.y; q2[4 * i + 3] = v.w;
        }
        // keys of token r (zero past the chunk), natural pair order of quarter c
        uint32_t ka[NP];
        if (r < tk.n) {
          if (tk.sink) {
            const float* kr = reinterpret_cast<const float*>(kst) + r * D + c * QD;
#pragma unroll
            for (int i = 0; i < NP / 2; ++i) {
              const float4 f = reinterpret_cast<const float4*>(kr)[i];
              ka[2 * i] = pack_half2(f.x, f.y);
              ka[2 * i + 1] = pack_half2(f.z, f.w);
            }
          } else {
            const uint8_t* kr = kst + (r * D + c * QD) * 2;
#pragma unroll
            for (int i = 0; i < NP / 4; ++i) {
              const uint4 v = reinterpret_cast<const uint4*>(kr)[i];
              ka[4 * i] = v.x; ka[4 * i + 1] = v.y; ka[4 * i + 2] = v.z; ka[4 * i + 3] = v.w;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < NP; ++i) ka[i] = 0u;
        }
        // scores: rows r = tokens, column 2c = head c (every column holds its head's q)
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < NKC; ++j) {
          if (j & 1) mma16816(acc1, ka[2 * j], 0u, ka[2 * j + 1], 0u, q2[2 * j], q2[2 * j + 1]);
          else       mma16816(acc0, ka[2 * j], 0u, ka[2 * j + 1], 0u, q2[2 * j], q2[2 * j + 1]);
        }
        s = (r < tk.n) ? (acc0[0] + acc1[0]) * (qscale * head_qf()) : -INFINITY;
      }
      if constexpr (MQ) {   // token r's position against column c's visible range
        const int64_t hi = col_hi(), lo = col_lo(hi);
        const int64_t t = tk.fresh ? f_fresh_pos(c_k)
                        : tk.sink  ? static_cast<int64_t>(tk.first) + r
                                   : g.S + a.plan.st.n_groups * g.G + tk.first + r;
        if (t > hi || (t >= g.S && t < lo)) s = -INFINITY;
      }
      const float mx = warp_max_rows(s);   // -inf only for a column that sees no token of the chunk
      if (mx > res_m + kRescale) {
        const float corr = (res_m == -INFINITY) ? 0.f : ex2(res_m - mx);
        res_m = mx;
        res_l *= corr;
        res_mn *= corr;
#pragma unroll
        for (int i = 0; i < NCT; ++i) { oacc[i][0] *= corr; oacc[i][1] *= corr; oacc[i][2] *= corr; oacc[i][3] *= corr; }
        rescale_corr(corr);
      }
      const float p = (MQ && s == -INFINITY) ? 0.f : ex2(s - res_m);
      res_l += p;
      {
        const float h = __uint_as_float(__float_as_uint(p) & 0xFFFFE000u);
        const __half hh = __float2half_rn(h), ll = __float2half_rn(p - h);
        *reinterpret_cast<__half*>(xw + xch_off<CH>(c, 0, r)) = hh;
        *reinterpret_cast<__half*>(xw + xch_off<CH>(c, 1, r)) = ll;
      }
      __syncwarp();
      // Oᵀ += Vᵀ P': B = P' of tokens 2c, 2c + 1 in column r (tokens 8.. are absent)
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xw + xch_off<CH>(hh_col, r & 1, 2 * c));
      const uint32_t tmask = (2 * c < tk.n ? 0x0000FFFFu : 0u) | (2 * c + 1 < tk.n ? 0xFFFF0000u : 0u);
      if (tk.sink) {
        const float* vr = reinterpret_cast<const float*>(vst);
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct) {
          uint32_t a0 = 0u, a1 = 0u;
          if (2 * c < tk.n) {
            const float* v0r = vr + (2 * c) * D + 16 * ct + r;
            const float x0 = v0r[0], y0 = (2 * c + 1 < tk.n) ? v0r[D] : 0.f;
            const float x1 = v0r[8], y1 = (2 * c + 1 < tk.n) ? v0r[D + 8] : 0.f;
            a0 = pack_half2(x0, y0);
            a1 = pack_half2(x1, y1);
          }
          mma16816(oacc[ct], a0, a1, 0u, 0u, b0, 0u);
        }
      } else {
        const uint32_t vbase = smem_addr(vst) + (lane & 7) * D * 2 + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct) {
          uint32_t a0, a1;
          ldsm_x2_trans(a0, a1, vbase + 32 * ct);
          mma16816(oacc[ct], a0 & tmask, a1 & tmask, 0u, 0u, b0, 0u);
        }
      }
      if (tk.fresh && (u_first + cu) % a.npass == 0) {
        // fused append: the token into its sink slot (widened to fp32) or its
        // ring slot; nothing this launch reads lives there
        uint8_t* base = const_cast<uint8_t*>(unit_base(u_first + cu));
        const int64_t fp = f_fresh_pos(c_k);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          for (int e = 4 * lane; e < D; e += 128) {
            const uint2 x = *reinterpret_cast<const uint2*>(kst + part * 16 * D + 2 * e);
            dbg_check_finite(g, make_uint4(x.x, x.y, 0u, 0u));
            if (fp < g.S) {
              const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
              const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
              uint8_t* dsk = base + (part ? g.sink_v : g.sink_k) + (fp * D + e) * 4;
              if (dbg_in_region(g, dsk, 16)) *reinterpret_cast<float4*>(dsk) = make_float4(f0.x, f0.y, f1.x, f1.y);
            } else {
              const int64_t slot = (fp - g.S) % g.R;
              uint8_t* drs = base + (part ? g.res_v : g.res_k) + (slot * D + e) * 2;
              if (dbg_in_region(g, drs, 8)) *reinterpret_cast<uint2*>(drs) = x;
            }
          }
        }
      }
      release();
    }
  }
  // the units not closed yet: the warp's last one, then those it had no work in
  while (cu < nunits) {
    if (cu >= 0) close_unit();
    ++cu;
    if (cu < nunits) open_unit(cu);
  }

  // drain this warp's copies still in flight (only after an abort), bounded
  // by the full limit whatever the consumer's was: the copies that were
  // issued land in this CTA's shared memory before it exits
  if (aborted) {
    for (int k = 0; k < inflight; ++k) {
      mbar_wait(bar0 + 8 * c_st, c_ph, kWaitNs);
      if (++c_st == a.ns) { c_st = 0; c_ph ^= 1u; }
    }
  }
}

// Uniform launches: the plan is the launch's own (one kernel parameter).
// HIO: q, out and the fresh token's rows are pinned host memory mapped into
// the device (the host-buffer entry points): the warps load the query and
// fresh rows with plain loads instead of bulk copies, and the merge writes
// the output to the host.
template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL = false, bool ROPE = false, bool HIO = false>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm) decode_mma_kernel(const Args a) {
  const NoRuns none{0};
  decode_body<D, BITS, CH, MQ, false, OUTL, ROPE, HIO>(a, none);
}

// Ragged launches: the runs' plans travel as a grid constant.
template <int D, int BITS, int CH, bool MQ, bool OUTL = false, bool ROPE = false, bool HIO = false>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm)
    decode_mma_ragged_kernel(const Args a, const __grid_constant__ RunTable rt) {
  decode_body<D, BITS, CH, MQ, true, OUTL, ROPE, HIO>(a, rt);
}

}  // namespace mma
}  // namespace kivi
