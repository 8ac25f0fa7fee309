// decode_b1.cu — the 1-bit (bit-stream) instantiations of the tensor-core decode kernel.
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_b1(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits<1>(a, grid, threads, smem, s);
}

int occupancy_b1(const Geo& g, int threads, int smem) { return occupancy_bits<1>(g, threads, smem); }

cudaError_t launch_rg_b1(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_bits_ragged<1>(a, rt, grid, threads, smem, s);
}

}  // namespace mma
}  // namespace kivi
