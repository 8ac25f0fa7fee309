// decode_simt_rope_d128.cu — the head-dim-128 instantiations of the CUDA-core
// decode kernel (decode_simt.cuh) for pre-RoPE keys, every code width.
#include "decode_simt.cuh"

namespace kivi {
namespace simt {

cudaError_t launch_rope_d128(const Args& a, int ctas, int smem, cudaStream_t s, int* resident) {
  return launch_rope_d<128>(a, ctas, smem, s, resident);
}

}  // namespace simt
}  // namespace kivi
