// stage.cu — one launch that gathers a step's inputs from pinned host memory
// into the arena's staging buffers, for the host-buffer entry points.
//
// Pinned host memory is mapped into the device's address space (unified
// addressing), so the kernel reads it directly with 16-byte loads over the
// chip-to-chip link: one launch in place of one host-to-device copy per
// input buffer, each of which pays its own setup latency.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

struct StageJob {
  const uint4* src[3];
  uint4* dst[3];
  int64_t n16[3];   // 16-byte chunks per buffer
};

__global__ void stage_kernel(const StageJob job) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
  for (int b = 0; b < 3; ++b)
    for (int64_t i = i0; i < job.n16[b]; i += stride) job.dst[b][i] = job.src[b][i];
}

}  // namespace

cudaError_t launch_stage(const void* const* src, void* const* dst, const int64_t* bytes, int n,
                         cudaStream_t stream) {
  StageJob job{};
  int64_t most = 0;
  for (int b = 0; b < 3; ++b) {
    if (b < n && bytes[b] > 0) {
      if (bytes[b] % 16 != 0) return cudaErrorInvalidValue;
      job.src[b] = static_cast<const uint4*>(src[b]);
      job.dst[b] = static_cast<uint4*>(dst[b]);
      job.n16[b] = bytes[b] / 16;
      if (job.n16[b] > most) most = job.n16[b];
    }
  }
  if (most == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (most + threads - 1) / threads;
  if (blocks > 304) blocks = 304;
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  stage_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(job);
  return cudaGetLastError();
}

}  // namespace kivi
