// decode.cu — host side of the split-K decode attention: launch shape,
// occupancy and the launch itself.  The kernel is in decode_mma.cuh (design
// notes there); decode_b{2,4,8}.cu instantiate it per code width.
#include "decode_launch.cuh"

namespace kivi {

namespace {
int32_t round_up32(int64_t x, int64_t a) { return static_cast<int32_t>((x + a - 1) / a * a); }
}  // namespace

DecodeShape decode_shape(const Geo& g) {
  DecodeShape sh{};
  const int64_t ch = (g.G % 32) == 0 ? 32 : 16;
  // a stage holds one group block, one tail chunk (4 fp32 or 8 fp16 tokens,
  // K and V) or the query rows of one head pass
  const int64_t chunk = 32 * static_cast<int64_t>(g.d);
  sh.stage_bytes = round_up32(g.block_bytes > chunk ? g.block_bytes : chunk, 128);
  // per warp besides its stages (mma::WarpSmem): query rows with padded
  // quarters, the combine slot, the P' exchange
  const int64_t q_bytes = 16 * (g.d / 2 + 16);
  const int64_t slot_bytes = 16 * (g.d + 4);
  const int64_t xch_bytes = ch == 32 ? 512 : 256;
  // with outlier tables: the [4][CH] p exchange and the [4][d] fp32 value corrections
  const int64_t corr_bytes = g.n_out > 0 ? 16 * (ch + g.d) : 0;
  // pre-RoPE keys: the angle row of the current group or tail chunk (mma::Rope)
  const int64_t rope_bytes = g.rope_l2b != 0.0 ? (g.d / 2 + 8) * 8 : 0;
  // shared memory of one CTA: the SM's 228 KB shared by kDecodeCtasPerSm
  // CTAs, less the 1 KB the driver reserves per CTA and room for the static
  // shared memory, and at most the 227 KB one CTA may have
  int64_t budget = (228 * 1024) / kDecodeCtasPerSm - 1024 - 512;
  if (budget > 227 * 1024 - 512) budget = 227 * 1024 - 512;
  auto per_warp_of = [&](int stages) {
    return static_cast<int64_t>(stages) * sh.stage_bytes + q_bytes + slot_bytes + xch_bytes + corr_bytes +
           rope_bytes + 12 * stages;
  };
  // as many warps (up to kDecodeWarps) as fit with two copy stages each, then
  // more stages (up to four) while they fit; very large group blocks get a
  // single stage rather than fewer than two warps
  int ns = 2;
  int64_t nw = budget / per_warp_of(ns);
  if (nw < 2) { ns = 1; nw = budget / per_warp_of(ns); }
  if (nw > kDecodeWarps) nw = kDecodeWarps;
  if (nw < 1) nw = 1;
  while (ns < 4 && nw * per_warp_of(ns + 1) <= budget) ++ns;
  const int64_t per_warp = per_warp_of(ns);
  sh.ns = ns;
  sh.nw = static_cast<int32_t>(nw);
  sh.smem_base = round_up32(nw * per_warp, 16);
  sh.npass = (g.rep + 3) / 4;
  return sh;
}

int decode_ctas_per_sm(const Geo& g) {
  const DecodeShape sh = decode_shape(g);
  const int threads = sh.nw * 32;
  const int smem = decode_smem(sh, g.split_stride);
  if (g.rope_l2b != 0.0) return mma::occupancy_rope_b(g.bits, g, threads, smem);
  if (g.n_out > 0) return mma::occupancy_outl_b(g.bits, g, threads, smem);
  if (g.bits == 2) return mma::occupancy_b2(g, threads, smem);
  if (g.bits == 4) return mma::occupancy_b4(g, threads, smem);
  if (g.bits == 8) return mma::occupancy_b8(g, threads, smem);
  return mma::occupancy_stream_b(g.bits, g, threads, smem);
}

cudaError_t launch_decode_scratch(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                  const DecodePlan& plan, float* partials, int32_t stride,
                                  unsigned* counters, unsigned* error, cudaStream_t stream) {
  if (plan.ctas < 1 || plan.tc < 1 || stride < 3) return cudaErrorInvalidValue;
  const DecodeShape sh = decode_shape(g);
  mma::Args a{};
  a.g = g;
  a.arena = arena;
  a.q = q;
  a.out = out;
  a.partials = partials;
  a.counters = counters;
  a.error = error;
  a.wait_ns = copy_wait_ns();
  a.plan = plan;
  a.ns = sh.ns;
  a.stage_bytes = sh.stage_bytes;
  a.stride = stride;
  if (plan.nq < 1 || plan.q_rows < plan.nq) return cudaErrorInvalidValue;
  a.npass = (plan.nq * g.rep + 3) / 4;   // head passes over the nq * rep query rows of a kv head
  a.units = g.B * g.hkv * a.npass;
  a.tc = plan.tc;
  a.uw = plan.n_vis_groups + plan.tc;
  // one wave of CTAs; each range holds at least one work position, and no unit
  // is shared by more CTAs than there are partial records (ceil(P/U) + 1 <= stride)
  int64_t ctas = plan.ctas;
  const int64_t work = static_cast<int64_t>(a.units) * a.uw;
  if (ctas > work) ctas = work;
  const int64_t cap = static_cast<int64_t>(stride - 2) * a.units;
  if (cap < 1) return cudaErrorInvalidValue;
  if (ctas > cap) ctas = cap;
  if (plan.q_rows > 1 && a.npass > 1) {
    // several query tokens: units are ordered pass-slowest, so in a grid of
    // P CTAs the passes of one group block are processed at P / npass CTAs
    // apart; when npass divides P they run at the same moment and L2 serves
    // all but the first read (npass / gcd(P, npass) DRAM reads otherwise).
    // The kernel is issue-bound, so the grid is trimmed to a multiple of
    // npass only when that keeps at least 95 % of the CTAs.
    const int64_t trimmed = ctas / a.npass * a.npass;
    if (trimmed > 0 && 20 * trimmed >= 19 * ctas) ctas = trimmed;
  }
  const dim3 grid(static_cast<unsigned>(ctas));
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  const int threads = sh.nw * 32;
  const int smem = decode_smem(sh, stride);
  if (g.rope_l2b != 0.0) return mma::launch_rope_b(g.bits, a, grid, threads, smem, stream);
  if (g.n_out > 0) return mma::launch_outl_b(g.bits, a, grid, threads, smem, stream);
  if (g.bits == 2) return mma::launch_b2(a, grid, threads, smem, stream);
  if (g.bits == 4) return mma::launch_b4(a, grid, threads, smem, stream);
  if (g.bits == 8) return mma::launch_b8(a, grid, threads, smem, stream);
  return mma::launch_stream_b(g.bits, a, grid, threads, smem, stream);
}

cudaError_t launch_decode_ragged(const Geo& g, const uint8_t* arena, const __half* q, __half* out,
                                 const DecodePlan& plan, const RunTable& runs, float* partials, int32_t stride,
                                 unsigned* counters, unsigned* error, cudaStream_t stream) {
  if (plan.ctas < 1 || stride < 3 || runs.n < 1 || runs.n > kMaxRuns || runs.W < 1) return cudaErrorInvalidValue;
  const DecodeShape sh = decode_shape(g);
  mma::Args a{};
  a.g = g;
  a.arena = arena;
  a.q = q;
  a.out = out;
  a.partials = partials;
  a.counters = counters;
  a.error = error;
  a.wait_ns = copy_wait_ns();
  a.plan = plan;
  a.plan.nq = 1;
  a.plan.q_rows = 1;
  a.ns = sh.ns;
  a.stage_bytes = sh.stage_bytes;
  a.stride = stride;
  a.npass = sh.npass;
  a.units = g.B * g.hkv * sh.npass;
  a.tc = 1;   // per run in the table
  a.uw = 1;
  int64_t ctas = plan.ctas;
  if (ctas > runs.W) ctas = runs.W;
  // a unit of w positions meets at most ceil(w P / W) + 1 of the P CTAs, which
  // must not exceed the stride of partial records: units of different widths
  // bound P by the widest one
  int64_t uw_max = 1;
  for (int k = 0; k < runs.n; ++k) uw_max = runs.r[k].uw > uw_max ? runs.r[k].uw : uw_max;
  const int64_t cap = static_cast<int64_t>(stride - 2) * runs.W / uw_max;
  if (cap < 1) return cudaErrorInvalidValue;
  if (ctas > cap) ctas = cap;
  const dim3 grid(static_cast<unsigned>(ctas));
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  const int threads = sh.nw * 32;
  const int smem = decode_smem(sh, stride);
  if (g.rope_l2b != 0.0) return mma::launch_rg_rope_b(g.bits, a, runs, grid, threads, smem, stream);
  if (g.n_out > 0) return mma::launch_rg_outl_b(g.bits, a, runs, grid, threads, smem, stream);
  if (g.bits == 2) return mma::launch_rg_b2(a, runs, grid, threads, smem, stream);
  if (g.bits == 4) return mma::launch_rg_b4(a, runs, grid, threads, smem, stream);
  if (g.bits == 8) return mma::launch_rg_b8(a, runs, grid, threads, smem, stream);
  return mma::launch_rg_stream_b(g.bits, a, runs, grid, threads, smem, stream);
}

cudaError_t launch_decode(const Geo& g, uint8_t* arena, const __half* q, __half* out,
                          const DecodePlan& plan, cudaStream_t stream) {
  return launch_decode_scratch(g, arena, q, out, plan, reinterpret_cast<float*>(arena + g.ws_partials),
                               g.split_stride, reinterpret_cast<unsigned*>(arena + g.ws_counters),
                               reinterpret_cast<unsigned*>(arena + g.ws_error), stream);
}

}  // namespace kivi
