// kivi_internal.cuh — geometry and kernel launchers shared by the CUDA
// translation units of libkivi.so.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kivi.h"

// Debug builds (compiled with -DKIVI_DEBUG_CHECKS=1 into libkivi_debug.so):
// the kernels check every arena address they derive against the handle's
// cache region and every input key, value and query for inf / NaN, and
// record what they find in the arena's error word (kErrIndex, kErrNonFinite)
// instead of trapping; an address that fails its check is not accessed.
// The product build compiles the checks out.
#ifndef KIVI_DEBUG_CHECKS
#define KIVI_DEBUG_CHECKS 0
#endif

namespace kivi {

constexpr bool kDebugChecks = KIVI_DEBUG_CHECKS != 0;
constexpr unsigned kErrIndex = 4u;       // (debug builds) a derived address left the cache region; skipped
constexpr unsigned kErrNonFinite = 8u;   // (debug builds) an input key, value or query was inf or NaN

// Everything a kernel needs to address the arena; passed by value.
struct Geo {
  int32_t bits, G, R, S, hq, hkv, d, B, rep;
  int64_t window, n_slots;
  int64_t unit_bytes, sink_k, sink_v, res_k, res_v, groups;
  int64_t block_bytes, blk_kq, blk_ks, blk_vq, blk_vs;
  int64_t blk_ko, blk_vo;  // outlier tables of a block: u16 row pointers [G + 1] by token,
                           // then from out_ent the 4-byte entries {u8 t, u8 c, fp16 x}
  int32_t n_out;           // entries per table; 0 without outliers
  int32_t out_ent;         // offset of the entries inside a table
  double rope_l2b;         // log2 of the RoPE base for pre-RoPE keys; 0 = keys arrive rotated
  int64_t cache_bytes;
  int64_t ws_partials;   // arena offset of the split-K partials
  int64_t ws_counters;   // arena offset of the per-unit merge counters
  int64_t ws_error;      // arena offset of the device error word
  int64_t ws_q, ws_out;  // arena offsets of the host-call staging buffers
  int64_t ws_k, ws_v;    // staging of one new token per sequence (fused host-buffer step)
  int64_t ws_rope;       // arena offset of the RoPE tables (pre-RoPE keys; rope.cu)
  int32_t max_splits;    // CTAs that may share one unit (partial records - 2)
  int32_t split_stride;  // partial records per query head
  // set when a handle opens: the handle's cache region [chk_lo, chk_hi) and
  // its error word (the debug checks; sub-geometries of a run keep them)
  const uint8_t* chk_lo;
  const uint8_t* chk_hi;
  unsigned* err;
};

// Debug checks (no-ops in the product build).
__device__ __forceinline__ bool dbg_in_region(const Geo& g, const void* p, int64_t bytes) {
  if constexpr (!kDebugChecks) return true;
  const uint8_t* q = static_cast<const uint8_t*>(p);
  if (q >= g.chk_lo && bytes >= 0 && q + bytes <= g.chk_hi) return true;
  atomicOr(g.err, kErrIndex);
  return false;
}
// eight fp16 values: an exponent field of all ones is inf or NaN
__device__ __forceinline__ void dbg_check_finite(const Geo& g, uint4 v) {
  if constexpr (kDebugChecks) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      bad |= (w[i] & 0x7C00u) == 0x7C00u || (w[i] & 0x7C000000u) == 0x7C000000u;
    if (bad) atomicOr(g.err, kErrNonFinite);
  }
}

// Cache state after T tokens (lazy flush: a token that reaches a full ring
// first pushes the ring's oldest G tokens out as one frozen group).
struct State {
  int64_t T, n_sink, n_groups, n_res;
};

__host__ __device__ inline State state_at(const Geo& g, int64_t T) {
  State s;
  s.T = T;
  s.n_sink = T < g.S ? T : g.S;
  const int64_t m = T > g.S ? T - g.S : 0;
  s.n_groups = (m <= g.R) ? 0 : (m - g.R + g.G - 1) / g.G;
  s.n_res = m - s.n_groups * g.G;
  return s;
}

// Host-side fault injection (kivi_debug_inject_launch_failure): true when
// the launch about to be made is the one armed to fail; it is then not made
// and the caller reports cudaErrorLaunchFailure.
bool injected_launch_failure();
// How long a decode warp waits for one of its copies before it gives up and
// sets the error word's copy bit (kivi_debug_set_wait_limit; 2 s by default).
unsigned long long copy_wait_ns();

// ---- pre-RoPE keys (rope.cu) ----
// Bytes of the RoPE tables of a geometry (0 without pre-RoPE keys), and the
// launch that writes them into the arena's workspace.
int64_t rope_table_bytes(const Geo& g);
cudaError_t launch_rope_table(const Geo& g, uint8_t* arena, cudaStream_t stream);

// ---- append (append.cu) ----
// Quantizes and packs groups [g_begin, g_end) of every unit.  Tokens with
// position < T_old come from the ring, the others from the new input, whose
// (sequence, kv head) rows hold n_stride tokens each.
cudaError_t launch_flush(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_stride, int64_t g_begin, int64_t g_end,
                         cudaStream_t stream);
// Writes new sink tokens [T_old, min(T_new, S)) and ring tokens
// [ring_begin, T_new) of every unit from the new input (T_new = T_old +
// n_new; rows of n_stride tokens).
// Copies n (at most 3) buffers of bytes[i] (multiples of 16, 16-byte aligned)
// from src[i] to dst[i] in one launch: the host-buffer entry points gather a
// step's inputs from pinned, device-mapped host memory this way (stage.cu).
cudaError_t launch_stage(const void* const* src, void* const* dst, const int64_t* bytes, int n,
                         cudaStream_t stream);
cudaError_t launch_write(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_new, int64_t n_stride, int64_t ring_begin, cudaStream_t stream);

// ---- decode (decode.cu) ----
struct DecodePlan {
  State st;               // the sinks and ring tokens read from the cache (st.T counts the fresh token)
  int64_t g_first;        // first frozen group that can hold a visible token
  int64_t n_vis_groups;   // groups [g_first, n_groups)
  int32_t tc;             // work positions (in groups) that stand for one unit's tail
  int32_t ctas;           // CTAs of the wave (the launch clamps it further)
  // fused append: one token per sequence attended straight from these
  // [B][H_kv][1][d] inputs and written by the kernel into the cache (at
  // position fresh_pos: a sink slot if below S, else its ring slot); null for
  // a plain decode
  const __half* k_fresh;
  const __half* v_fresh;
  int64_t fresh_pos;
  // query tokens per sequence: 1 for a decode; M for the causal attention of
  // a chunk's M newest tokens, query j at position q_pos0 + j (q and out are
  // then [B][M][H_q][d])
  int32_t nq;
  int32_t q_rows;         // query tokens per sequence in the q and out buffers (>= nq)
  int64_t q_pos0;
  // 1: q, out, k_fresh and v_fresh are pinned host memory mapped into the
  // device (the host-buffer entry points, word-rule widths without outlier
  // tables or pre-RoPE keys): the host-io kernel instantiations read the
  // query and fresh rows with plain loads and write the output to the host
  int32_t host_io;
};

// Ragged launches: one decode launch over sequences of different lengths.
// The batch is cut into runs of consecutive sequences of equal length; each
// run's plan travels in the kernel's parameters (a grid constant, read with
// constant loads).  Units keep the uniform numbering (sequence, kv head,
// head pass), so run k holds units [ubase, ubase + nb * h_kv * npass); their
// work positions start at pos0, uw per unit.
struct RunPlan {
  int64_t pos0;        // first work position of the run's units
  int64_t g_first;     // first frozen group that can hold a visible token
  int64_t q_pos0;      // position of the query (T - 1)
  int64_t fresh_pos;   // fused step: position of the appended token
  int32_t ubase;       // first unit of the run
  int32_t uw;          // work positions per unit
  int32_t n_vis;       // visible frozen groups per unit
  int32_t n_sink;      // sink tokens read from the cache
  int32_t n_res;       // ring tokens read from the cache
  int32_t rs0;         // ring slot of the oldest ring token
  uint32_t slot0;      // slot of the first visible group
  int32_t b0, nb;      // the run's sequences
  int32_t pad;
};
constexpr int kMaxRuns = 64;
struct RunTable {
  int32_t n;           // runs
  int32_t pad;
  int64_t W;           // work positions of the launch
  RunPlan r[kMaxRuns];
};
struct NoRuns {
  int32_t n;
};

// Decode launch shape: up to kDecodeWarps warps per CTA and kDecodeCtasPerSm
// CTAs per SM (the kernel's launch bounds; registers per thread follow).
constexpr int kDecodeWarps = 8;
constexpr int kDecodeCtasPerSm = 2;

// Launch shape of the decode kernel for a geometry (host side, no device work).
struct DecodeShape {
  int32_t nw;             // warps per CTA
  int32_t ns;             // copy stages per warp
  int32_t stage_bytes;
  int32_t smem_base;      // dynamic shared memory per CTA
  int32_t npass;          // head passes (4 query heads each) per kv head
};
DecodeShape decode_shape(const Geo& g);
// Dynamic shared memory of one CTA (independent of the partial-record stride).
inline int32_t decode_smem(const DecodeShape& sh, int32_t /*stride*/) { return sh.smem_base; }
// Resident decode CTAs per SM for this geometry (queries the device).
int decode_ctas_per_sm(const Geo& g);

// Packing rule of a code width: the word rule (b in {2, 4, 8}) or a bit stream.
inline bool word_rule(int bits) { return bits == 2 || bits == 4 || bits == 8; }

// Decode with the arena's own workspace for the split-K partials.
cudaError_t launch_decode(const Geo& g, uint8_t* arena, const __half* q, __half* out,
                          const DecodePlan& plan, cudaStream_t stream);
// Decode with caller-chosen scratch: `partials` holds B * nq * h_q * stride
// records of (d + 4) floats, `counters` ceil(nq * rep / 4) words per
// (sequence, kv head),
// zero on entry and left zero on exit, `error` one word that the kernel ORs
// with 1 if a copy never arrived.
cudaError_t launch_decode_scratch(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                  const DecodePlan& plan, float* partials, int32_t stride,
                                  unsigned* counters, unsigned* error, cudaStream_t stream);
// One decode launch over the runs of `runs` (plan: the launch-wide fields
// nq = q_rows = 1, ctas, k_fresh / v_fresh for a fused step; runs: per-run
// plans with pos0, ubase and W filled in by the caller).
cudaError_t launch_decode_ragged(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                 const DecodePlan& plan, const RunTable& runs, float* partials, int32_t stride,
                                 unsigned* counters, unsigned* error, cudaStream_t stream);
// The fused step's flush over a ragged batch: for each sequence b whose next
// token (at position T_old[b], from the [B][h_kv][1][d] inputs) reaches a
// full ring, the ring's oldest G tokens become its next frozen group; the
// other sequences' blocks return at once.  T_old by run (b0, nb, fresh_pos).
cudaError_t launch_flush_ragged(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                                const RunTable& runs, cudaStream_t stream);

}  // namespace kivi
