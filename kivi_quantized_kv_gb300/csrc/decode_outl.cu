// decode_outl.cu — dispatch of the decode with outlier corrections to its
// per-width instantiations (decode_outl_b{2,3,4}.cu).
#include "decode_outl.cuh"

namespace kivi {
namespace mma {

#define KIVI_OUTL_DECL(B)                                                                                      \
  cudaError_t launch_outl_b##B(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);               \
  cudaError_t launch_rg_outl_b##B(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,         \
                                  cudaStream_t s);                                                             \
  int occupancy_outl_b##B(const Geo& g, int threads, int smem);
KIVI_OUTL_DECL(2)
KIVI_OUTL_DECL(3)
KIVI_OUTL_DECL(4)
#undef KIVI_OUTL_DECL

cudaError_t launch_outl_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  switch (bits) {
    case 2: return launch_outl_b2(a, grid, threads, smem, s);
    case 3: return launch_outl_b3(a, grid, threads, smem, s);
    case 4: return launch_outl_b4(a, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rg_outl_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                             cudaStream_t s) {
  switch (bits) {
    case 2: return launch_rg_outl_b2(a, rt, grid, threads, smem, s);
    case 3: return launch_rg_outl_b3(a, rt, grid, threads, smem, s);
    case 4: return launch_rg_outl_b4(a, rt, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_outl_b(int bits, const Geo& g, int threads, int smem) {
  switch (bits) {
    case 2: return occupancy_outl_b2(g, threads, smem);
    case 3: return occupancy_outl_b3(g, threads, smem);
    case 4: return occupancy_outl_b4(g, threads, smem);
    default: return 1;
  }
}

}  // namespace mma
}  // namespace kivi
