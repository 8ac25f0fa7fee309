// decode_b6.cu — the 6-bit (bit-stream) instantiations of the tensor-core decode kernel.
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_b6(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits<6>(a, grid, threads, smem, s);
}

int occupancy_b6(const Geo& g, int threads, int smem) { return occupancy_bits<6>(g, threads, smem); }

cudaError_t launch_rg_b6(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits_ragged<6>(a, rt, grid, threads, smem, s);
}

}  // namespace mma
}  // namespace kivi
