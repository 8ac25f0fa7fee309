// decode_outl_b2.cu — the 2-bit instantiations of the decode with outlier
// corrections.
#include "decode_outl.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_outl_b2(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  const NoRuns none{0};
  return launch_outl<2, false>(a, none, grid, threads, smem, s);
}

cudaError_t launch_rg_outl_b2(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_outl<2, true>(a, rt, grid, threads, smem, s);
}

int occupancy_outl_b2(const Geo& g, int threads, int smem) { return occupancy_outl<2>(g, threads, smem); }

}  // namespace mma
}  // namespace kivi
