// decode_outl.cuh — launch of the tensor-core decode with outlier
// corrections (the OUTL instantiations): 32-token chunks and one query token
// per sequence; head dim 64 or 128 for the word widths, 128 for 3 bits.
// Each decode_outl_b*.cu instantiates one code width.
#pragma once

#include "decode_launch.cuh"

namespace kivi {
namespace mma {

template <int BITS, bool RG>
cudaError_t launch_outl(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  if (a.plan.q_rows > 1 || (a.g.G % 32) != 0) return cudaErrorInvalidValue;
  if constexpr (stream_bits<BITS>()) {
    if (a.g.d != 128) return cudaErrorInvalidValue;
    return launch_one<128, BITS, 32, false, RG, true>(a, rt, grid, threads, smem, s);
  } else {
    return a.g.d == 64 ? launch_one<64, BITS, 32, false, RG, true>(a, rt, grid, threads, smem, s)
                       : launch_one<128, BITS, 32, false, RG, true>(a, rt, grid, threads, smem, s);
  }
}

template <int BITS>
int occupancy_outl(const Geo& g, int threads, int smem) {
  if (stream_bits<BITS>() || g.d == 128) return occupancy_one<128, BITS, 32, false, false, true>(threads, smem);
  if constexpr (!stream_bits<BITS>()) return occupancy_one<64, BITS, 32, false, false, true>(threads, smem);
  return 1;
}

}  // namespace mma
}  // namespace kivi
