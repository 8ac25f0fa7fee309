// decode_simt.cu — host side of the CUDA-core decode for the bit-stream code
// widths: split count and launch.  The kernel is in decode_simt.cuh (design
// notes there); decode_simt_d{64,128}.cu instantiate it per head dim.
#include "decode_simt.cuh"

namespace kivi {

cudaError_t launch_decode_simt(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                               const DecodePlan& plan, float* partials, int32_t stride, unsigned* counters,
                               int32_t sms, cudaStream_t stream) {
  if ((g.G != 32 && g.G != 64) || g.rep > simt::kMaxRep || stride < 3) return cudaErrorInvalidValue;
  simt::Args a{};
  a.g = g;
  a.arena = arena;
  a.q = q;
  a.out = out;
  a.partials = partials;
  a.counters = counters;
  a.plan = plan;
  a.stride = stride;
  a.sink_items = static_cast<int32_t>((plan.st.n_sink + simt::kTail - 1) / simt::kTail);
  a.items = static_cast<int32_t>(plan.n_vis_groups) + a.sink_items +
            static_cast<int32_t>((plan.st.n_res + simt::kTail - 1) / simt::kTail);
  if (a.items < 1) a.items = 1;
  const int64_t units = static_cast<int64_t>(g.B) * g.hkv;
  const int smem = simt::kWarps * (g.d == 64 ? simt::Smem<64>::bytes(g) : simt::Smem<128>::bytes(g)) +
                   simt::rope_bytes(g);
  // many short CTAs (about eight per resident slot) so that the waves end
  // evenly, within the partial records a unit has
  int resident = 1;
  cudaError_t e = g.d == 64 ? simt::launch_d64(a, 0, smem, stream, &resident)
                            : simt::launch_d128(a, 0, smem, stream, &resident);
  if (e != cudaSuccess) return e;
  const int64_t want = static_cast<int64_t>(sms) * (resident > 0 ? resident : 1) * 8;
  int64_t splits = (want + units - 1) / units;
  if (splits > a.items) splits = a.items;
  if (splits > stride) splits = stride;
  if (splits < 1) splits = 1;
  a.splits = static_cast<int32_t>(splits);
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  const int ctas = static_cast<int>(units * splits);
  return g.d == 64 ? simt::launch_d64(a, ctas, smem, stream, nullptr)
                   : simt::launch_d128(a, ctas, smem, stream, nullptr);
}

}  // namespace kivi
