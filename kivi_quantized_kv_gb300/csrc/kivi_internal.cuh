// kivi_internal.cuh — geometry and kernel launchers shared by the CUDA
// translation units of libkivi.so.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kivi.h"

namespace kivi {

// Everything a kernel needs to address the arena; passed by value.
struct Geo {
  int32_t bits, G, R, S, hq, hkv, d, B, rep;
  int64_t window, n_slots;
  int64_t unit_bytes, sink_k, sink_v, res_k, res_v, groups;
  int64_t block_bytes, blk_kq, blk_ks, blk_vq, blk_vs;
  int64_t cache_bytes;
  int64_t ws_partials;   // arena offset of the split-K partials
  int64_t ws_counters;   // arena offset of the per-unit merge counters
  int64_t ws_q, ws_out;  // arena offsets of the host-call staging buffers
  int32_t max_splits;
};

// Cache state after T tokens (lazy flush: a token that reaches a full ring
// first pushes the ring's oldest G tokens out as one frozen group).
struct State {
  int64_t T, n_sink, n_groups, n_res;
};

inline State state_at(const Geo& g, int64_t T) {
  State s;
  s.T = T;
  s.n_sink = T < g.S ? T : g.S;
  const int64_t m = T > g.S ? T - g.S : 0;
  s.n_groups = (m <= g.R) ? 0 : (m - g.R + g.G - 1) / g.G;
  s.n_res = m - s.n_groups * g.G;
  return s;
}

// ---- append (append.cu) ----
// Quantizes and packs groups [g_begin, g_end) of every unit.  Tokens with
// position < T_old come from the ring, the others from the new input.
cudaError_t launch_flush(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_new, int64_t g_begin, int64_t g_end,
                         cudaStream_t stream);
// Writes new sink tokens [T_old, min(T_new, S)) and ring tokens
// [ring_begin, T_new) of every unit from the new input.
cudaError_t launch_write(const Geo& g, uint8_t* arena, const __half* k_new, const __half* v_new,
                         int64_t T_old, int64_t n_new, int64_t ring_begin, cudaStream_t stream);

// ---- decode (decode.cu) ----
struct DecodePlan {
  State st;
  int64_t g_first;        // first frozen group that can hold a visible token
  int64_t n_vis_groups;   // groups [g_first, n_groups)
  int32_t splits;         // split-K partitions per unit
  int32_t groups_per_split;
};

// Decode with the arena's own workspace for the split-K partials.
cudaError_t launch_decode(const Geo& g, uint8_t* arena, const __half* q, __half* out,
                          const DecodePlan& plan, cudaStream_t stream);
// Decode with caller-chosen scratch: `partials` holds B * h_q * max_splits
// records of (d + 2) floats, `counters` one word per (sequence, kv head).
cudaError_t launch_decode_scratch(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                  const DecodePlan& plan, float* partials, unsigned* counters,
                                  cudaStream_t stream);

}  // namespace kivi
