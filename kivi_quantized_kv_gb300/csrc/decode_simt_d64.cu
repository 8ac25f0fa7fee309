// decode_simt_d64.cu — the head-dim-64 instantiations of the CUDA-core decode
// kernel (decode_simt.cuh), one translation unit per head dim so they build
// in parallel.
#include "decode_simt.cuh"

namespace kivi {
namespace simt {

cudaError_t launch_d64(const Args& a, int ctas, int smem, cudaStream_t s, int* resident) {
  return launch_d<64>(a, ctas, smem, s, resident);
}

}  // namespace simt
}  // namespace kivi
