// decode_rope.cu — dispatch of the decode for pre-RoPE keys to its per-width
// instantiations (decode_rope_b{1..8}.cu).
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

#define KIVI_ROPE_DECL(B)                                                                                       \
  cudaError_t launch_rope_b##B(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);                \
  cudaError_t launch_rg_rope_b##B(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,          \
                                  cudaStream_t s);                                                              \
  int occupancy_rope_b##B(const Geo& g, int threads, int smem);
KIVI_ROPE_DECL(1)
KIVI_ROPE_DECL(2)
KIVI_ROPE_DECL(3)
KIVI_ROPE_DECL(4)
KIVI_ROPE_DECL(5)
KIVI_ROPE_DECL(6)
KIVI_ROPE_DECL(7)
KIVI_ROPE_DECL(8)
#undef KIVI_ROPE_DECL

cudaError_t launch_rope_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  switch (bits) {
    case 1: return launch_rope_b1(a, grid, threads, smem, s);
    case 2: return launch_rope_b2(a, grid, threads, smem, s);
    case 3: return launch_rope_b3(a, grid, threads, smem, s);
    case 4: return launch_rope_b4(a, grid, threads, smem, s);
    case 5: return launch_rope_b5(a, grid, threads, smem, s);
    case 6: return launch_rope_b6(a, grid, threads, smem, s);
    case 7: return launch_rope_b7(a, grid, threads, smem, s);
    case 8: return launch_rope_b8(a, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rg_rope_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                             cudaStream_t s) {
  switch (bits) {
    case 1: return launch_rg_rope_b1(a, rt, grid, threads, smem, s);
    case 2: return launch_rg_rope_b2(a, rt, grid, threads, smem, s);
    case 3: return launch_rg_rope_b3(a, rt, grid, threads, smem, s);
    case 4: return launch_rg_rope_b4(a, rt, grid, threads, smem, s);
    case 5: return launch_rg_rope_b5(a, rt, grid, threads, smem, s);
    case 6: return launch_rg_rope_b6(a, rt, grid, threads, smem, s);
    case 7: return launch_rg_rope_b7(a, rt, grid, threads, smem, s);
    case 8: return launch_rg_rope_b8(a, rt, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_rope_b(int bits, const Geo& g, int threads, int smem) {
  switch (bits) {
    case 1: return occupancy_rope_b1(g, threads, smem);
    case 2: return occupancy_rope_b2(g, threads, smem);
    case 3: return occupancy_rope_b3(g, threads, smem);
    case 4: return occupancy_rope_b4(g, threads, smem);
    case 5: return occupancy_rope_b5(g, threads, smem);
    case 6: return occupancy_rope_b6(g, threads, smem);
    case 7: return occupancy_rope_b7(g, threads, smem);
    case 8: return occupancy_rope_b8(g, threads, smem);
    default: return 1;
  }
}

}  // namespace mma
}  // namespace kivi
