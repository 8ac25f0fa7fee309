// decode_outl.cuh — launch of the tensor-core decode with outlier
// corrections (the OUTL instantiations): 32-token chunks, head dim 64 or 128,
// one query token per sequence or (uniform launches) several.
// Each decode_outl_b*.cu instantiates one code width.
#pragma once

#include "decode_launch.cuh"

namespace kivi {
namespace mma {

template <int BITS, bool MQ, bool RG>
cudaError_t launch_outl_mq(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem,
                           cudaStream_t s) {
  return a.g.d == 64 ? launch_one<64, BITS, 32, MQ, RG, true>(a, rt, grid, threads, smem, s)
                     : launch_one<128, BITS, 32, MQ, RG, true>(a, rt, grid, threads, smem, s);
}

// the decode (and fused step, uniform or ragged) and, uniform only, the
// multi-query attention of chunked prefill
template <int BITS, bool RG>
cudaError_t launch_outl(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  if ((a.g.G % 32) != 0) return cudaErrorInvalidValue;
  if constexpr (RG) {
    if (a.plan.q_rows > 1) return cudaErrorInvalidValue;
    return launch_outl_mq<BITS, false, true>(a, rt, grid, threads, smem, s);
  } else {
    return a.plan.q_rows > 1 ? launch_outl_mq<BITS, true, false>(a, rt, grid, threads, smem, s)
                             : launch_outl_mq<BITS, false, false>(a, rt, grid, threads, smem, s);
  }
}

template <int BITS>
int occupancy_outl(const Geo& g, int threads, int smem) {
  return g.d == 64 ? occupancy_one<64, BITS, 32, false, false, true>(threads, smem)
                   : occupancy_one<128, BITS, 32, false, false, true>(threads, smem);
}

}  // namespace mma
}  // namespace kivi
