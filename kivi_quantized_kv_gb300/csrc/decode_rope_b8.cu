// decode_rope_b8.cu — the 8-bit instantiations of the tensor-core decode for
// pre-RoPE keys.
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_rope_b8(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_rope_bits<8>(a, grid, threads, smem, s);
}
cudaError_t launch_rg_rope_b8(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  return launch_rope_bits_ragged<8>(a, rt, grid, threads, smem, s);
}
int occupancy_rope_b8(const Geo& g, int threads, int smem) { return occupancy_rope_bits<8>(g, threads, smem); }

}  // namespace mma
}  // namespace kivi
