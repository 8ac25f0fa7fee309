// decode_stream.cu — dispatch of the bit-stream code widths (1, 3, 5, 6, 7) to
// their tensor-core decode instantiations (decode_b{1,3,5,6,7}.cu).
#include "decode_launch.cuh"

namespace kivi {
namespace mma {

cudaError_t launch_b1(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b3(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b5(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b6(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b7(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
int occupancy_b1(const Geo& g, int threads, int smem);
int occupancy_b3(const Geo& g, int threads, int smem);
int occupancy_b5(const Geo& g, int threads, int smem);
int occupancy_b6(const Geo& g, int threads, int smem);
int occupancy_b7(const Geo& g, int threads, int smem);
cudaError_t launch_rg_b1(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b3(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b5(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b6(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b7(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);

cudaError_t launch_stream_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  switch (bits) {
    case 1: return launch_b1(a, grid, threads, smem, s);
    case 3: return launch_b3(a, grid, threads, smem, s);
    case 5: return launch_b5(a, grid, threads, smem, s);
    case 6: return launch_b6(a, grid, threads, smem, s);
    case 7: return launch_b7(a, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rg_stream_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                               cudaStream_t s) {
  switch (bits) {
    case 1: return launch_rg_b1(a, rt, grid, threads, smem, s);
    case 3: return launch_rg_b3(a, rt, grid, threads, smem, s);
    case 5: return launch_rg_b5(a, rt, grid, threads, smem, s);
    case 6: return launch_rg_b6(a, rt, grid, threads, smem, s);
    case 7: return launch_rg_b7(a, rt, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_stream_b(int bits, const Geo& g, int threads, int smem) {
  switch (bits) {
    case 1: return occupancy_b1(g, threads, smem);
    case 3: return occupancy_b3(g, threads, smem);
    case 5: return occupancy_b5(g, threads, smem);
    case 6: return occupancy_b6(g, threads, smem);
    case 7: return occupancy_b7(g, threads, smem);
    default: return 1;
  }
}

}  // namespace mma
}  // namespace kivi
