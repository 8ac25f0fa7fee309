// decode_launch.cuh — per-instantiation launch and occupancy helpers of the
// tensor-core decode kernel; each decode_b*.cu instantiates one bit width.
#pragma once

#include <atomic>

#include "decode_mma.cuh"

namespace kivi {
namespace mma {

// the kernel of an instantiation
template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL = false, bool ROPE = false, bool HIO = false>
constexpr auto kernel_of() {
  if constexpr (RG) return decode_mma_ragged_kernel<D, BITS, CH, MQ, OUTL, ROPE, HIO>;
  else return decode_mma_kernel<D, BITS, CH, MQ, false, OUTL, ROPE, HIO>;
}

template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL = false, bool ROPE = false, bool HIO = false>
cudaError_t prepare() {
  // opt in to the largest dynamic shared memory once per instantiation
  static std::atomic<int> done{0};
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kernel_of<D, BITS, CH, MQ, RG, OUTL, ROPE, HIO>());
  if (e != cudaSuccess) return e;
  // the opt-in limit covers static + dynamic shared memory
  e = cudaFuncSetAttribute(kernel_of<D, BITS, CH, MQ, RG, OUTL, ROPE, HIO>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - static_cast<int>(fa.sharedSizeBytes));
  if (e == cudaSuccess) done.store(1, std::memory_order_release);
  return e;
}

template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL = false, bool ROPE = false, bool HIO = false>
cudaError_t launch_one(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  cudaError_t e = prepare<D, BITS, CH, MQ, RG, OUTL, ROPE, HIO>();
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the CTAs may start (and set up their
  // shared memory) while the previous kernel in the stream drains; the kernel
  // waits for that kernel's completion before it touches global memory
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (RG) e = cudaLaunchKernelEx(&cfg, kernel_of<D, BITS, CH, MQ, RG, OUTL, ROPE, HIO>(), a, rt);
  else e = cudaLaunchKernelEx(&cfg, kernel_of<D, BITS, CH, MQ, RG, OUTL, ROPE, HIO>(), a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int BITS, int CH, bool MQ, bool RG, bool OUTL = false, bool ROPE = false>
int occupancy_one(int threads, int smem) {
  if (prepare<D, BITS, CH, MQ, RG, OUTL, ROPE>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_of<D, BITS, CH, MQ, RG, OUTL, ROPE>(), threads, smem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// one instantiation per (head dim, chunk of the group, several query tokens,
// ragged)
template <int BITS, bool MQ, bool RG, bool HIO = false>
cudaError_t launch_mq(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  const bool ch32 = (a.g.G % 32) == 0;
  if (a.g.d == 64)
    return ch32 ? launch_one<64, BITS, 32, MQ, RG, false, false, HIO>(a, rt, grid, threads, smem, s)
                : launch_one<64, BITS, 16, MQ, RG, false, false, HIO>(a, rt, grid, threads, smem, s);
  return ch32 ? launch_one<128, BITS, 32, MQ, RG, false, false, HIO>(a, rt, grid, threads, smem, s)
              : launch_one<128, BITS, 16, MQ, RG, false, false, HIO>(a, rt, grid, threads, smem, s);
}

// bit-stream widths: 32-token chunks only (a lane's 8 codes of a value row
// start on a 32-bit word); at head dim 64 a lane's quarter of a key row may
// start on a 16-bit boundary, which the kernel aligns
template <int BITS, bool MQ, bool RG>
cudaError_t launch_stream(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  if ((a.g.G % 32) != 0) return cudaErrorInvalidValue;
  return a.g.d == 64 ? launch_one<64, BITS, 32, MQ, RG>(a, rt, grid, threads, smem, s)
                     : launch_one<128, BITS, 32, MQ, RG>(a, rt, grid, threads, smem, s);
}

template <int BITS>
cudaError_t launch_bits(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  const NoRuns none{0};
  // the single-query instantiation assumes one query token per sequence row
  if constexpr (stream_bits<BITS>()) {
    return a.plan.q_rows > 1 ? launch_stream<BITS, true, false>(a, none, grid, threads, smem, s)
                             : launch_stream<BITS, false, false>(a, none, grid, threads, smem, s);
  } else {
    // host-io instantiations: the word-rule widths, one query token
    if (a.plan.host_io && a.plan.q_rows == 1) return launch_mq<BITS, false, false, true>(a, none, grid, threads, smem, s);
    return a.plan.q_rows > 1 ? launch_mq<BITS, true, false>(a, none, grid, threads, smem, s)
                             : launch_mq<BITS, false, false>(a, none, grid, threads, smem, s);
  }
}

// ragged launches: one query token per sequence (decode and the fused step)
template <int BITS>
cudaError_t launch_bits_ragged(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                               cudaStream_t s) {
  if constexpr (stream_bits<BITS>()) return launch_stream<BITS, false, true>(a, rt, grid, threads, smem, s);
  else if (a.plan.host_io) return launch_mq<BITS, false, true, true>(a, rt, grid, threads, smem, s);
  else return launch_mq<BITS, false, true>(a, rt, grid, threads, smem, s);
}

// the other instantiations have the same launch bounds and shared memory
template <int BITS>
int occupancy_bits(const Geo& g, int threads, int smem) {
  if constexpr (stream_bits<BITS>()) {
    return g.d == 64 ? occupancy_one<64, BITS, 32, false, false>(threads, smem)
                     : occupancy_one<128, BITS, 32, false, false>(threads, smem);
  } else {
    const bool ch32 = (g.G % 32) == 0;
    if (g.d == 64)
      return ch32 ? occupancy_one<64, BITS, 32, false, false>(threads, smem)
                  : occupancy_one<64, BITS, 16, false, false>(threads, smem);
    return ch32 ? occupancy_one<128, BITS, 32, false, false>(threads, smem)
                : occupancy_one<128, BITS, 16, false, false>(threads, smem);
  }
}

// pre-RoPE keys (decode_rope_b*.cu): every width, 32-token chunks (G 32 or
// 64), head dims 64 and 128; one or several query tokens, uniform or ragged
template <int BITS, bool MQ, bool RG>
cudaError_t launch_rope_mq(const Args& a, const RunTableT<RG>& rt, dim3 grid, int threads, int smem, cudaStream_t s) {
  if ((a.g.G % 32) != 0) return cudaErrorInvalidValue;
  return a.g.d == 64 ? launch_one<64, BITS, 32, MQ, RG, false, true>(a, rt, grid, threads, smem, s)
                     : launch_one<128, BITS, 32, MQ, RG, false, true>(a, rt, grid, threads, smem, s);
}
template <int BITS>
cudaError_t launch_rope_bits(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s) {
  const NoRuns none{0};
  return a.plan.q_rows > 1 ? launch_rope_mq<BITS, true, false>(a, none, grid, threads, smem, s)
                           : launch_rope_mq<BITS, false, false>(a, none, grid, threads, smem, s);
}
template <int BITS>
cudaError_t launch_rope_bits_ragged(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                                    cudaStream_t s) {
  return launch_rope_mq<BITS, false, true>(a, rt, grid, threads, smem, s);
}
template <int BITS>
int occupancy_rope_bits(const Geo& g, int threads, int smem) {
  return g.d == 64 ? occupancy_one<64, BITS, 32, false, false, false, true>(threads, smem)
                   : occupancy_one<128, BITS, 32, false, false, false, true>(threads, smem);
}
cudaError_t launch_rope_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_rope_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                             cudaStream_t s);
int occupancy_rope_b(int bits, const Geo& g, int threads, int smem);

// defined in decode_b2.cu, decode_b4.cu, decode_b8.cu
cudaError_t launch_b2(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b4(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_b8(const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b2(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b4(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_b8(const Args& a, const RunTable& rt, dim3 grid, int threads, int smem, cudaStream_t s);
// the bit-stream widths (decode_b1.cu, decode_b3.cu, decode_b5.cu, decode_b6.cu, decode_b7.cu)
cudaError_t launch_stream_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_stream_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                               cudaStream_t s);
int occupancy_stream_b(int bits, const Geo& g, int threads, int smem);
int occupancy_b2(const Geo& g, int threads, int smem);
// with outlier tables (decode_outl.cu): 2 to 4 bits, 32-token chunks, one
// or (uniform launches) several query tokens per sequence
cudaError_t launch_outl_b(int bits, const Args& a, dim3 grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_rg_outl_b(int bits, const Args& a, const RunTable& rt, dim3 grid, int threads, int smem,
                             cudaStream_t s);
int occupancy_outl_b(int bits, const Geo& g, int threads, int smem);
int occupancy_b4(const Geo& g, int threads, int smem);
int occupancy_b8(const Geo& g, int threads, int smem);

}  // namespace mma
}  // namespace kivi
