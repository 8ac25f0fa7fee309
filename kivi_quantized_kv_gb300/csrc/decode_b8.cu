// decode_b8.cu — the 8-bit instantiations of the tensor-core decode kernel.
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_b8(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits<8>(a, grid, threads, smem, s);
}

int occupancy_b8(const Geo& g, int threads, int smem) { return occupancy_bits<8>(g, threads, smem); }

cudaError_t launch_rg_b8(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits_ragged<8>(a, rt, grid, threads, smem, s);
}

}  // namespace mma
}  // namespace kivi
