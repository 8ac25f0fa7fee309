// kivi_host.cu — the C ABI of libkivi.so (declared in include/kivi.h).
//
// Host-side work only: parameter checks, the arena layout, the token counters
// (the cache state is a pure function of the token count T), the choice of
// split-K partitions, and kernel launches.  No device memory is allocated,
// freed or synchronised here.
#include "kivi_internal.cuh"

#include <atomic>
#include <mutex>
#include <new>
#include <vector>

namespace kivi {
namespace {
std::atomic<int64_t> g_fail_countdown{0};   // 0 = disarmed; n = the n-th launch from now fails
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
}  // namespace
unsigned long long copy_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
bool injected_launch_failure() {
  int64_t n = g_fail_countdown.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_fail_countdown.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return n == 1;
  }
  return false;
}
}  // namespace kivi

struct kivi_cache {
  kivi_params p;
  kivi::Geo g;
  uint8_t* arena;
  size_t arena_bytes;
  std::vector<int64_t> T;   // tokens appended so far, per sequence
  int32_t forced_splits;
  int32_t num_sms;
  int32_t ctas_per_sm;   // resident decode CTAs per SM for this geometry
};

namespace {

using kivi::Geo;
using kivi::State;

constexpr int64_t kAlign = 256;
constexpr int kMaxRep = 8;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate(const kivi_params* p) {
  if (!p) return KIVI_ENULL;
  if (p->bits < 1 || p->bits > 8) return KIVI_EINVAL;
  // the bit-stream widths: a value row of a 32-token chunk is whole 32-bit
  // words; groups of 32 or 64 tokens
  if (!kivi::word_rule(p->bits) && p->group != 32 && p->group != 64) return KIVI_EINVAL;
  if (!(p->head_dim == 64 || p->head_dim == 128)) return KIVI_EINVAL;
  if (p->group < 16 || p->group > 256 || p->group % 16 != 0) return KIVI_EINVAL;
  if (p->residual < p->group || p->residual % p->group != 0) return KIVI_EINVAL;
  if (p->residual > (1 << 20)) return KIVI_EINVAL;
  if (p->sinks < 0 || p->sinks > 1024) return KIVI_EINVAL;
  if (p->h_kv < 1 || p->h_q < 1 || p->h_q % p->h_kv != 0) return KIVI_EINVAL;
  if (p->h_q / p->h_kv > kMaxRep) return KIVI_EINVAL;
  if (p->batch < 1 || p->batch > 65535) return KIVI_EINVAL;
  if (static_cast<int64_t>(p->h_kv) * ((p->h_q / p->h_kv + 3) / 4) > 65535) return KIVI_EINVAL;
  if (p->window < 0 || p->max_tokens < 0) return KIVI_EINVAL;
  if (p->window > 0 && p->window < p->residual) return KIVI_EINVAL;
  if (p->outlier_permille < 0 || p->outlier_permille > 50 || p->reserved != 0) return KIVI_EINVAL;
  // the outlier corrections are built into the tensor-core decode at 2 to 4
  // bits with 32-token chunks
  if (p->outlier_permille > 0 && (p->bits < 2 || p->bits > 4 || p->group % 32 != 0)) return KIVI_EINVAL;
  // pre-RoPE keys: 32-token chunks (a key's rotation pairs sit in one lane's
  // two regions; value rows whole 32-bit words), without outlier tables
  if (!(p->rope_base == 0.0 || (p->rope_base > 1.0 && p->rope_base <= 1e7))) return KIVI_EINVAL;
  if (p->rope_base != 0.0 && ((p->group != 32 && p->group != 64) || p->outlier_permille != 0)) return KIVI_EINVAL;
  return KIVI_OK;
}

// CTAs that may share one (sequence, kv head, head pass) unit: the decode
// launches at most kMaxDecodeCtas CTAs (one wave on any GPU with up to 256
// SMs at 4 CTAs each), cut into equal ranges over the units' work, so a unit
// meets at most ceil(kMaxDecodeCtas / units) + 1 of them.
constexpr int64_t kMaxDecodeCtas = 1024;
int32_t max_splits_for(const kivi_params& p) {
  const int64_t units = static_cast<int64_t>(p.batch) * p.h_kv * ((p.h_q / p.h_kv + 3) / 4);
  return static_cast<int32_t>((kMaxDecodeCtas + units - 1) / units + 1);
}

Geo geometry(const kivi_params& p) {
  Geo g{};
  g.bits = p.bits; g.G = p.group; g.R = p.residual; g.S = p.sinks;
  g.hq = p.h_q; g.hkv = p.h_kv; g.d = p.head_dim; g.B = p.batch; g.rep = p.h_q / p.h_kv;
  g.window = p.window;
  g.rope_l2b = p.rope_base != 0.0 ? std::log2(p.rope_base) : 0.0;
  const int64_t d = p.head_dim, G = p.group, b = p.bits;
  if (p.window > 0) {
    g.n_slots = (p.window + G - 1) / G + 1;
  } else {
    g.n_slots = kivi::state_at(g, p.max_tokens).n_groups;
  }
  g.sink_k = 0;
  g.sink_v = g.sink_k + p.sinks * d * 4;
  g.res_k = g.sink_v + p.sinks * d * 4;
  g.res_v = g.res_k + p.residual * d * 2;
  g.groups = g.res_v + p.residual * d * 2;
  g.blk_kq = 0;
  g.blk_ks = g.blk_kq + G * d * b / 8;
  g.blk_vq = g.blk_ks + 2 * d * 2;
  g.blk_vs = g.blk_vq + d * G * b / 8;
  g.n_out = static_cast<int32_t>((static_cast<int64_t>(p.outlier_permille) * G * d + 999) / 1000);
  g.out_ent = g.n_out ? static_cast<int32_t>(((G + 1) * 2 + 3) / 4 * 4) : 0;
  const int64_t table = g.n_out ? (g.out_ent + 4 * static_cast<int64_t>(g.n_out) + 15) / 16 * 16 : 0;
  g.blk_ko = g.blk_vs + G * 2 * 2;
  g.blk_vo = g.blk_ko + table;
  g.block_bytes = g.blk_vo + table;
  g.unit_bytes = g.groups + g.n_slots * g.block_bytes;
  g.cache_bytes = static_cast<int64_t>(p.batch) * p.h_kv * g.unit_bytes;
  g.max_splits = max_splits_for(p);
  g.split_stride = g.max_splits + 2;
  const int64_t bhq = static_cast<int64_t>(p.batch) * p.h_q;
  const int64_t npass = (g.rep + 3) / 4;
  g.ws_partials = round_up(g.cache_bytes, kAlign);
  g.ws_counters = round_up(g.ws_partials + bhq * g.split_stride * (d + 4) * 4, kAlign);
  g.ws_error = round_up(g.ws_counters + static_cast<int64_t>(p.batch) * p.h_kv * npass * 4, kAlign);
  g.ws_q = round_up(g.ws_error + 4, kAlign);
  g.ws_out = round_up(g.ws_q + bhq * d * 2, kAlign);
  const int64_t bhkv = static_cast<int64_t>(p.batch) * p.h_kv;
  g.ws_k = round_up(g.ws_out + bhq * d * 2, kAlign);
  g.ws_v = round_up(g.ws_k + bhkv * d * 2, kAlign);
  g.ws_rope = round_up(g.ws_v + bhkv * d * 2, kAlign);
  return g;
}

int64_t arena_bytes_of(const Geo& g) { return round_up(g.ws_rope + kivi::rope_table_bytes(g), kAlign); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KIVI_OK : KIVI_ECUDA; }

// Sequences may hold different token counts (ragged batches).  Every call
// works on runs of consecutive sequences that share their token count (and,
// for the ragged calls, their count of new tokens or queries): a run is a
// batch of its own for the kernels, addressed through a geometry with B = nb
// and the cache region shifted to its first sequence (a unit's bytes do not
// depend on its sequence index).  A batch of equal lengths is one run.
struct Run {
  int32_t b0, nb;   // sequences [b0, b0 + nb)
  int64_t T, n;     // their token count and per-call count (0 when unused)
};

// Runs of equal (T[b], n_of(b)).
template <class F>
std::vector<Run> runs_of(const kivi_cache& c, F n_of) {
  std::vector<Run> out;
  for (int32_t b = 0; b < c.g.B; ++b) {
    const int64_t n = n_of(b);
    if (!out.empty() && out.back().T == c.T[b] && out.back().n == n) {
      out.back().nb += 1;
    } else {
      out.push_back(Run{b, 1, c.T[b], n});
    }
  }
  return out;
}
std::vector<Run> runs_of(const kivi_cache& c) {
  return runs_of(c, [](int32_t) { return int64_t{0}; });
}

Geo sub_geo(const Geo& g, int32_t nb) {
  Geo s = g;
  s.B = nb;
  return s;
}
uint8_t* run_base(const kivi_cache& c, const Run& r) {
  return c.arena + static_cast<int64_t>(r.b0) * c.g.hkv * c.g.unit_bytes;
}
int64_t max_tokens_of(const kivi_cache& c) {
  int64_t m = 0;
  for (const int64_t t : c.T) m = t > m ? t : m;
  return m;
}
int64_t min_tokens_of(const kivi_cache& c) {
  int64_t m = c.T.empty() ? 0 : c.T[0];
  for (const int64_t t : c.T) m = t < m ? t : m;
  return m;
}

// First frozen group that can hold a visible token, and the plan of splits,
// for nb sequences of T tokens each and nq query tokens per sequence at
// positions T - nq .. T - 1 (1 for a decode), whose q and out rows are
// q_rows tokens apart per sequence.
kivi::DecodePlan plan_for(const kivi_cache& c, int64_t T, int32_t nb, int32_t nq = 1, int32_t q_rows = 1) {
  kivi::DecodePlan pl{};
  pl.st = kivi::state_at(c.g, T);
  pl.nq = nq;
  pl.q_rows = q_rows;
  pl.q_pos0 = T - nq;
  int64_t first = pl.st.n_groups - c.g.n_slots;
  if (first < 0) first = 0;
  if (c.g.window > 0) {
    const int64_t lo = pl.q_pos0 + 1 - c.g.window;       // first position the oldest query sees
    if (lo > c.g.S) {
      const int64_t gl = (lo - c.g.S) / c.g.G;            // group holding position lo
      if (gl > first) first = gl;
    }
  }
  if (first > pl.st.n_groups) first = pl.st.n_groups;
  pl.g_first = first;
  pl.n_vis_groups = pl.st.n_groups - first;
  // one wave of resident CTAs; the sinks are cut into chunks of 4 tokens and
  // the ring into chunks of 8, one work position each (at least one position,
  // empty when the cache is)
  int64_t ctas = static_cast<int64_t>(c.num_sms) * c.ctas_per_sm;
  if (ctas > kMaxDecodeCtas) ctas = kMaxDecodeCtas;
  if (c.forced_splits > 0) {   // a fixed number of CTAs per unit
    const int64_t units = static_cast<int64_t>(nb) * c.g.hkv * ((static_cast<int64_t>(nq) * c.g.rep + 3) / 4);
    ctas = units * c.forced_splits;
  }
  pl.ctas = static_cast<int32_t>(ctas > 0 ? ctas : 1);
  const int64_t tc = (pl.st.n_sink + 3) / 4 + (pl.st.n_res + 7) / 8;
  pl.tc = static_cast<int32_t>(tc < 1 ? 1 : tc);
  return pl;
}

}  // namespace

extern "C" {

size_t kivi_cache_bytes(const kivi_params* params) {
  if (validate(params) != KIVI_OK) return 0;
  return static_cast<size_t>(arena_bytes_of(geometry(*params)));
}

}  // extern "C"

namespace {
// A handle over an arena; the cache region is zeroed (a new cache) or kept
// (restore), the workspace's counters and error word are always cleared.
int open_handle(const kivi_params* params, void* d_arena, size_t arena_bytes, const int64_t* tokens, bool keep,
                void* cuda_stream, kivi_cache** out) {
  if (!out || !d_arena) return KIVI_ENULL;
  const int v = validate(params);
  if (v != KIVI_OK) return v;
  if (!aligned(d_arena, kAlign)) return KIVI_EALIGN;
  const Geo g = geometry(*params);
  if (static_cast<int64_t>(arena_bytes) < arena_bytes_of(g)) return KIVI_ENOSPC;
  if (keep) {
    for (int32_t b = 0; b < params->batch; ++b)
      if (tokens[b] < 0 || (params->window == 0 && tokens[b] > params->max_tokens)) return KIVI_EINVAL;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KIVI_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KIVI_ECUDA;
  kivi_cache* c = new (std::nothrow) kivi_cache();
  if (!c) return KIVI_ENULL;
  c->p = *params;
  c->g = g;
  c->g.chk_lo = static_cast<const uint8_t*>(d_arena);
  c->g.chk_hi = c->g.chk_lo + g.cache_bytes;
  c->g.err = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(d_arena) + g.ws_error);
  c->arena = static_cast<uint8_t*>(d_arena);
  c->arena_bytes = arena_bytes;
  try {
    c->T.assign(static_cast<size_t>(params->batch), 0);
  } catch (...) {
    delete c;
    return KIVI_ENULL;
  }
  if (keep) c->T.assign(tokens, tokens + params->batch);
  c->forced_splits = 0;
  c->num_sms = sms > 0 ? sms : 1;
  c->ctas_per_sm = kivi::decode_ctas_per_sm(g);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const int64_t from = keep ? g.ws_counters : 0;   // counters and error word are adjacent
  const int64_t to = keep ? g.ws_error + 4 : arena_bytes_of(g);
  cudaError_t e = cudaMemsetAsync(c->arena + from, 0, static_cast<size_t>(to - from), s);
  if (e == cudaSuccess) e = kivi::launch_rope_table(g, c->arena, s);   // pre-RoPE keys: the rotation tables
  if (e != cudaSuccess) { delete c; return KIVI_ECUDA; }
  *out = c;
  return KIVI_OK;
}
}  // namespace

extern "C" {

int kivi_cache_create(const kivi_params* params, void* d_arena, size_t arena_bytes, void* cuda_stream,
                      kivi_cache** out) {
  return open_handle(params, d_arena, arena_bytes, nullptr, false, cuda_stream, out);
}

int kivi_cache_restore(const kivi_params* params, void* d_arena, size_t arena_bytes, const int64_t* tokens,
                       void* cuda_stream, kivi_cache** out) {
  if (!tokens) return KIVI_ENULL;
  return open_handle(params, d_arena, arena_bytes, tokens, true, cuda_stream, out);
}

int kivi_debug_inject_launch_failure(int64_t n) {
  if (n < 0) return KIVI_EINVAL;
  kivi::g_fail_countdown.store(n, std::memory_order_relaxed);
  return KIVI_OK;
}

int kivi_debug_set_wait_limit(int64_t ns) {
  if (ns < 0) return KIVI_EINVAL;
  kivi::g_wait_ns.store(ns == 0 ? kivi::kDefaultWaitNs : static_cast<unsigned long long>(ns),
                        std::memory_order_relaxed);
  return KIVI_OK;
}

void kivi_cache_destroy(kivi_cache* cache) { delete cache; }

}  // extern "C"

namespace {

// Appends n tokens to every sequence of run r (its token count r.T) from
// inputs whose (sequence, kv head) rows hold n_stride tokens.
cudaError_t append_run(const kivi_cache& c, const Run& r, const __half* k_new, const __half* v_new, int64_t n,
                       int64_t n_stride, cudaStream_t s) {
  const Geo gs = sub_geo(c.g, r.nb);
  const int64_t T_old = r.T, T_new = r.T + n;
  const State s0 = kivi::state_at(gs, T_old), s1 = kivi::state_at(gs, T_new);
  const int64_t in = static_cast<int64_t>(r.b0) * gs.hkv * n_stride * gs.d;
  uint8_t* base = run_base(c, r);
  // groups created by this append; with a window only the last n_slots survive
  int64_t g_begin = s0.n_groups;
  if (s1.n_groups - gs.n_slots > g_begin) g_begin = s1.n_groups - gs.n_slots;
  cudaError_t e = kivi::launch_flush(gs, base, k_new + in, v_new + in, T_old, n_stride, g_begin, s1.n_groups, s);
  if (e != cudaSuccess) return e;
  // the ring keeps the last R tokens of the stream (flushed or not)
  int64_t ring_begin = T_old;
  if (ring_begin < gs.S) ring_begin = gs.S;
  if (T_new - gs.R > ring_begin) ring_begin = T_new - gs.R;
  if (ring_begin > T_new) ring_begin = T_new;
  return kivi::launch_write(gs, base, k_new + in, v_new + in, T_old, n, n_stride, ring_begin, s);
}

// The attention of run r: q and out rows of its first sequence at
// b0 * q_rows * h_q; scratch pointers absolute.
cudaError_t attn_run(const kivi_cache& c, const Run& r, const kivi::DecodePlan& pl, const __half* q, __half* out,
                     float* partials, int32_t stride, unsigned* counters, unsigned* error, cudaStream_t s) {
  const Geo gs = sub_geo(c.g, r.nb);
  const int64_t row0 = static_cast<int64_t>(r.b0) * pl.q_rows * gs.hq * gs.d;
  return kivi::launch_decode_scratch(gs, run_base(c, r), q + row0, out + row0, pl, partials, stride, counters,
                                     error, s);
}
float* ws_partials(const kivi_cache& c) { return reinterpret_cast<float*>(c.arena + c.g.ws_partials); }

// The plans of runs [first, first + count) for one ragged launch (one query
// token per sequence); fused: every sequence also attends to and appends one
// new token taken from the inputs.
kivi::RunTable run_table(const kivi_cache& c, const std::vector<Run>& runs, size_t first, size_t count,
                         bool fused) {
  const Geo& g = c.g;
  const int64_t npass = (g.rep + 3) / 4;
  kivi::RunTable t{};
  t.n = static_cast<int32_t>(count);
  int64_t pos = 0;
  for (size_t i = 0; i < count; ++i) {
    const Run& r = runs[first + i];
    kivi::DecodePlan pl = plan_for(c, fused ? r.T + 1 : r.T, r.nb);
    int64_t tc = pl.tc;
    if (fused) {   // the fresh token is a tail chunk of its own, not read from the cache
      if (r.T < g.S) pl.st.n_sink -= 1; else pl.st.n_res -= 1;
      tc = (pl.st.n_sink + 3) / 4 + (pl.st.n_res + 7) / 8 + 1;
    }
    kivi::RunPlan& rp = t.r[i];
    rp.pos0 = pos;
    rp.g_first = pl.g_first;
    rp.q_pos0 = pl.q_pos0;
    rp.fresh_pos = r.T;
    rp.ubase = static_cast<int32_t>(r.b0 * g.hkv * npass);
    rp.n_vis = static_cast<int32_t>(pl.n_vis_groups);
    rp.uw = static_cast<int32_t>(pl.n_vis_groups + tc);
    rp.n_sink = static_cast<int32_t>(pl.st.n_sink);
    rp.n_res = static_cast<int32_t>(pl.st.n_res);
    rp.rs0 = static_cast<int32_t>((pl.st.n_groups * g.G) % g.R);
    rp.slot0 = static_cast<uint32_t>(g.window > 0 ? pl.g_first % g.n_slots : pl.g_first);
    rp.b0 = r.b0;
    rp.nb = r.nb;
    pos += static_cast<int64_t>(r.nb) * g.hkv * npass * rp.uw;
  }
  t.W = pos;
  return t;
}

// Decode (fused: append one token from k_fresh / v_fresh first) over every
// sequence: one launch when all lengths agree, else one ragged launch per
// kMaxRuns runs (fused: preceded by one flush launch when a run freezes a
// group).
cudaError_t decode_all(const kivi_cache& c, const __half* q, __half* out, const __half* k_fresh,
                       const __half* v_fresh, float* partials, int32_t stride, unsigned* counters,
                       unsigned* error, cudaStream_t s, bool host_io = false) {
  const Geo& g = c.g;
  const bool fused = k_fresh != nullptr;
  const std::vector<Run> runs = runs_of(c);
  if (runs.size() == 1) {
    const Run& r = runs[0];
    if (fused) {
      const State s0 = kivi::state_at(g, r.T), s1 = kivi::state_at(g, r.T + 1);
      if (s1.n_groups > s0.n_groups) {
        // the token reaches a full ring: its oldest G tokens freeze first, as
        // in kivi_append (a launch of its own, before the decode reads them)
        int64_t g_begin = s0.n_groups;
        if (s1.n_groups - g.n_slots > g_begin) g_begin = s1.n_groups - g.n_slots;
        const cudaError_t e = kivi::launch_flush(g, c.arena, k_fresh, v_fresh, r.T, 1, g_begin, s1.n_groups, s);
        if (e != cudaSuccess) return e;
      }
    }
    kivi::DecodePlan pl = plan_for(c, fused ? r.T + 1 : r.T, r.nb);
    if (fused) {
      // the fresh token is attended straight from the inputs (and written into
      // its sink or ring slot by the same launch), so the cache's own tail is
      // one token shorter
      if (r.T < g.S) pl.st.n_sink -= 1; else pl.st.n_res -= 1;
      pl.tc = static_cast<int32_t>((pl.st.n_sink + 3) / 4 + (pl.st.n_res + 7) / 8 + 1);
      pl.k_fresh = k_fresh;
      pl.v_fresh = v_fresh;
      pl.fresh_pos = r.T;
    }
    pl.host_io = host_io ? 1 : 0;
    return attn_run(c, r, pl, q, out, partials, stride, counters, error, s);
  }
  for (size_t first = 0; first < runs.size(); first += kivi::kMaxRuns) {
    const size_t count = runs.size() - first < static_cast<size_t>(kivi::kMaxRuns) ? runs.size() - first
                                                                                     : kivi::kMaxRuns;
    const kivi::RunTable t = run_table(c, runs, first, count, fused);
    if (fused) {
      bool freezes = false;
      for (size_t i = first; i < first + count; ++i)
        freezes = freezes || kivi::state_at(g, runs[i].T + 1).n_groups > kivi::state_at(g, runs[i].T).n_groups;
      if (freezes) {
        const cudaError_t e = kivi::launch_flush_ragged(g, c.arena, k_fresh, v_fresh, t, s);
        if (e != cudaSuccess) return e;
      }
    }
    kivi::DecodePlan pl = plan_for(c, runs[first].T, g.B);   // launch-wide fields: the grid
    pl.k_fresh = k_fresh;
    pl.v_fresh = v_fresh;
    pl.host_io = host_io ? 1 : 0;
    const cudaError_t e = kivi::launch_decode_ragged(g, c.arena, q, out, pl, t, partials, stride, counters, error, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
unsigned* ws_counters(const kivi_cache& c) { return reinterpret_cast<unsigned*>(c.arena + c.g.ws_counters); }
// The host-io decode instantiations exist for the word-rule widths without
// outlier tables or pre-RoPE keys (the other caches gather through stage.cu).
bool host_io_kernels(const Geo& g) { return kivi::word_rule(g.bits) && g.n_out == 0 && g.rope_l2b == 0.0; }
// The device address of a pinned host buffer mapped into the device's address
// space (cudaHostAlloc, cudaMallocHost or cudaHostRegister under unified
// addressing), or null for any other pointer (pageable host memory included).
const void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();   // not a pointer CUDA knows: clear the error
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
  return at.devicePointer;
}
unsigned* ws_error(const kivi_cache& c) { return reinterpret_cast<unsigned*>(c.arena + c.g.ws_error); }

}  // namespace

extern "C" {

int kivi_append(kivi_cache* c, const void* k_new, const void* v_new, int64_t n, void* cuda_stream) {
  if (!c || !k_new || !v_new) return KIVI_ENULL;
  if (n < 1) return KIVI_EINVAL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return KIVI_EALIGN;
  if (c->g.window == 0 && max_tokens_of(*c) + n > c->p.max_tokens) return KIVI_ECAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  for (const Run& r : runs_of(*c)) {
    const cudaError_t e = append_run(*c, r, static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                     n, n, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  for (int64_t& t : c->T) t += n;
  return KIVI_OK;
}

int kivi_append_ragged(kivi_cache* c, const void* k_new, const void* v_new, const int64_t* n_tokens,
                       int64_t n_max, void* cuda_stream) {
  if (!c || !k_new || !v_new || !n_tokens) return KIVI_ENULL;
  if (n_max < 1) return KIVI_EINVAL;
  for (int32_t b = 0; b < c->g.B; ++b) {
    if (n_tokens[b] < 0 || n_tokens[b] > n_max) return KIVI_EINVAL;
    if (c->g.window == 0 && c->T[b] + n_tokens[b] > c->p.max_tokens) return KIVI_ECAPACITY;
  }
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return KIVI_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  for (const Run& r : runs_of(*c, [&](int32_t b) { return n_tokens[b]; })) {
    if (r.n == 0) continue;
    const cudaError_t e = append_run(*c, r, static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                     r.n, n_max, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  for (int32_t b = 0; b < c->g.B; ++b) c->T[b] += n_tokens[b];
  return KIVI_OK;
}

int kivi_cache_tokens(const kivi_cache* c, int64_t* tokens) {
  if (!c || !tokens) return KIVI_ENULL;
  for (int32_t b = 0; b < c->g.B; ++b) tokens[b] = c->T[b];
  return KIVI_OK;
}

int kivi_decode_attn(kivi_cache* c, const void* q, void* out, void* cuda_stream) {
  if (!c || !q || !out) return KIVI_ENULL;
  if (!aligned(q, 16) || !aligned(out, 16)) return KIVI_EALIGN;
  return cuda_status(decode_all(*c, static_cast<const __half*>(q), static_cast<__half*>(out), nullptr, nullptr,
                                ws_partials(*c), c->g.split_stride, ws_counters(*c), ws_error(*c),
                                static_cast<cudaStream_t>(cuda_stream)));
}

int kivi_append_decode_attn(kivi_cache* c, const void* k_new, const void* v_new, const void* q, void* out,
                            void* cuda_stream) {
  if (!c || !k_new || !v_new || !q || !out) return KIVI_ENULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(q, 16) || !aligned(out, 16)) return KIVI_EALIGN;
  const Geo& g = c->g;
  if (g.window == 0 && max_tokens_of(*c) + 1 > c->p.max_tokens) return KIVI_ECAPACITY;
  const cudaError_t e = decode_all(*c, static_cast<const __half*>(q), static_cast<__half*>(out),
                                   static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                   ws_partials(*c), g.split_stride, ws_counters(*c), ws_error(*c),
                                   static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_status(e);
  for (int64_t& t : c->T) t += 1;
  return KIVI_OK;
}

int kivi_append_decode_attn_host(kivi_cache* c, const void* k_host, const void* v_host, const void* q_host,
                                 void* out_host, void* cuda_stream) {
  if (!c || !k_host || !v_host || !q_host || !out_host) return KIVI_ENULL;
  const Geo& g = c->g;
  if (g.window == 0 && max_tokens_of(*c) + 1 > c->p.max_tokens) return KIVI_ECAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const size_t q_bytes = static_cast<size_t>(g.B) * g.hq * g.d * 2;
  const size_t kv_bytes = static_cast<size_t>(g.B) * g.hkv * g.d * 2;
  void* dk = c->arena + g.ws_k;
  void* dv = c->arena + g.ws_v;
  void* dq = c->arena + g.ws_q;
  void* dout = c->arena + g.ws_out;
  // pinned host buffers mapped into the device's address space: one launch
  // gathers the inputs into the staging area and the decode writes its
  // output straight to out_host; other host memory: a copy per buffer
  const void* mk = mapped_host(k_host);
  const void* mv = mapped_host(v_host);
  const void* mq = mapped_host(q_host);
  void* mo = const_cast<void*>(mapped_host(out_host));
  const bool mapped = mk && mv && mq && mo && aligned(mk, 16) && aligned(mv, 16) && aligned(mq, 16) &&
                      aligned(mo, 16);
  if (mapped && host_io_kernels(g)) {
    // the decode's host-io instantiation reads q and the fresh rows itself
    const cudaError_t e = decode_all(*c, static_cast<const __half*>(mq), static_cast<__half*>(mo),
                                     static_cast<const __half*>(mk), static_cast<const __half*>(mv),
                                     ws_partials(*c), g.split_stride, ws_counters(*c), ws_error(*c), s, true);
    if (e != cudaSuccess) return cuda_status(e);
    for (int64_t& t : c->T) t += 1;
    return KIVI_OK;
  }
  if (mapped) {
    const void* src[3] = {mk, mv, mq};
    void* dst[3] = {dk, dv, dq};
    const int64_t bytes[3] = {static_cast<int64_t>(kv_bytes), static_cast<int64_t>(kv_bytes),
                              static_cast<int64_t>(q_bytes)};
    const cudaError_t e = kivi::launch_stage(src, dst, bytes, 3, s);
    if (e != cudaSuccess) return cuda_status(e);
    return kivi_append_decode_attn(c, dk, dv, dq, mo, cuda_stream);
  }
  if (cudaMemcpyAsync(dk, k_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dv, v_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dq, q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return KIVI_ECUDA;
  const int st = kivi_append_decode_attn(c, dk, dv, dq, dout, cuda_stream);
  if (st != KIVI_OK) return st;
  return cuda_status(cudaMemcpyAsync(out_host, dout, q_bytes, cudaMemcpyDeviceToHost, s));
}

int kivi_decode_attn_host(kivi_cache* c, const void* q_host, void* out_host, void* cuda_stream) {
  if (!c || !q_host || !out_host) return KIVI_ENULL;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const size_t bytes = static_cast<size_t>(c->g.B) * c->g.hq * c->g.d * 2;
  void* dq = c->arena + c->g.ws_q;
  void* dout = c->arena + c->g.ws_out;
  const void* mq = mapped_host(q_host);
  void* mo = const_cast<void*>(mapped_host(out_host));
  if (mq && mo && aligned(mq, 16) && aligned(mo, 16) && host_io_kernels(c->g))
    return cuda_status(decode_all(*c, static_cast<const __half*>(mq), static_cast<__half*>(mo), nullptr, nullptr,
                                  ws_partials(*c), c->g.split_stride, ws_counters(*c), ws_error(*c), s, true));
  if (mq && mo && aligned(mq, 16) && aligned(mo, 16)) {   // as kivi_append_decode_attn_host
    const void* src[1] = {mq};
    void* dst[1] = {dq};
    const int64_t nb[1] = {static_cast<int64_t>(bytes)};
    const cudaError_t e = kivi::launch_stage(src, dst, nb, 1, s);
    if (e != cudaSuccess) return cuda_status(e);
    return kivi_decode_attn(c, dq, mo, cuda_stream);
  }
  cudaError_t e = cudaMemcpyAsync(dq, q_host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return KIVI_ECUDA;
  const int st = kivi_decode_attn(c, dq, dout, cuda_stream);
  if (st != KIVI_OK) return st;
  e = cudaMemcpyAsync(out_host, dout, bytes, cudaMemcpyDeviceToHost, s);
  return cuda_status(e);
}

// ---------------------------------------------------------------------------
// Decode without any device allocation by anyone: the split-K scratch lives in
// a fixed, library-owned device array instead of the caller's arena
// workspace.  For callers that hand this library only their input and output
// buffers and cannot obtain more device memory while decoding, e.g. a plugin
// running inside a host runtime that owns all device memory and forbids
// allocation during execution, or a latency-critical loop where cudaMalloc's
// implicit device synchronisation is unacceptable.
//
// The array is a module-scope __device__ variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits (the CUDA
// driver materialises it when it loads the variable, which with lazy module
// loading happens at the latest on the first call on that device).  In host
// code the symbol is only a host-side stand-in, never a device address, so its
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, on the first call made on that device (make that first
// call before any stream capture).  All calls share the array and it keeps the
// previous call's contents: the merge counters are cleared on every call, and
// calls whose work overlaps on the GPU (other streams, other host threads)
// race on it.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KIVI_ECUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return KIVI_EINVAL;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KIVI_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KIVI_OK;
}

}  // namespace

int kivi_decode_attn_noalloc(kivi_cache* c, const void* q, void* out, void* cuda_stream) {
  if (!c || !q || !out) return KIVI_ENULL;
  if (!aligned(q, 16) || !aligned(out, 16)) return KIVI_EALIGN;
  // scratch: [merge counters, npass per (sequence, kv head)][partials]; the
  // bounded waits report into the cache's own error word (kivi_read_error)
  const int64_t npass = (c->g.rep + 3) / 4;
  const int64_t head_bytes = round_up(static_cast<int64_t>(c->g.B) * c->g.hkv * npass * 4, kAlign);
  const int64_t record = static_cast<int64_t>(c->g.B) * c->g.hq * (c->g.d + 4) * 4;   // one CTA per unit
  const int64_t fit = (static_cast<int64_t>(kNoAllocScratchBytes) - head_bytes) / record;
  if (fit < 3) return KIVI_ESCRATCH;   // at least two CTAs per unit
  void* base = nullptr;
  const int st = noalloc_scratch(&base);
  if (st != KIVI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  unsigned char* bytes = static_cast<unsigned char*>(base);
  unsigned* counters = reinterpret_cast<unsigned*>(bytes);
  float* partials = reinterpret_cast<float*>(bytes + head_bytes);
  if (cudaMemsetAsync(bytes, 0, static_cast<size_t>(head_bytes), s) != cudaSuccess) return KIVI_ECUDA;
  // each launch leaves the counters zero and caps its CTAs so a unit's
  // partials fit
  return cuda_status(decode_all(*c, static_cast<const __half*>(q), static_cast<__half*>(out), nullptr, nullptr,
                                partials, static_cast<int32_t>(fit), counters, ws_error(*c), s));
}

int kivi_set_num_splits(kivi_cache* c, int32_t num_splits) {
  if (!c) return KIVI_ENULL;
  if (num_splits < 0) return KIVI_EINVAL;
  c->forced_splits = num_splits;
  return KIVI_OK;
}

namespace {
// the geometry fields of a layout (the state fields are left 0)
kivi_layout layout_of_geo(const Geo& g) {
  kivi_layout L{};
  L.n_slots = g.n_slots;
  L.sink_k = g.sink_k; L.sink_v = g.sink_v; L.res_k = g.res_k; L.res_v = g.res_v; L.groups = g.groups;
  L.block_bytes = g.block_bytes; L.blk_kq = g.blk_kq; L.blk_ks = g.blk_ks; L.blk_vq = g.blk_vq; L.blk_vs = g.blk_vs;
  L.blk_ko = g.blk_ko; L.blk_vo = g.blk_vo; L.n_outliers = g.n_out; L.out_entries = g.out_ent;
  L.unit_bytes = g.unit_bytes; L.cache_bytes = g.cache_bytes;
  L.workspace_offset = g.ws_partials;
  L.arena_bytes = arena_bytes_of(g);
  L.workspace_bytes = L.arena_bytes - g.ws_partials;
  L.max_splits = g.max_splits;
  return L;
}
}  // namespace

int kivi_layout_for(const kivi_params* p, kivi_layout* out) {
  if (!p || !out) return KIVI_ENULL;
  const int v = validate(p);
  if (v != KIVI_OK) return v;
  *out = layout_of_geo(geometry(*p));
  return KIVI_OK;
}

int kivi_cache_layout(const kivi_cache* c, kivi_layout* out) {
  if (!c || !out) return KIVI_ENULL;
  const Geo& g = c->g;
  const State st = kivi::state_at(g, c->T[0]);
  bool uniform = true;
  for (const int64_t t : c->T) uniform = uniform && t == c->T[0];
  kivi_layout L = layout_of_geo(g);
  // the state of sequence 0; tokens is -1 when the sequences' lengths differ
  L.tokens = uniform ? c->T[0] : -1; L.n_sink = st.n_sink; L.n_groups = st.n_groups; L.n_res = st.n_res;
  *out = L;
  return KIVI_OK;
}

namespace {
// Algorithmic bytes of one attention call over run r with nq query tokens
// per sequence: the cache bytes the union of the queries' visible sets
// needs, plus q and out (fp16).
int64_t attn_bytes(const kivi_cache& c, const Run& r, int64_t nq) {
  const Geo& g = c.g;
  const kivi::DecodePlan pl = plan_for(c, r.T, r.nb, static_cast<int32_t>(nq));
  const int64_t d = g.d;
  const int64_t lo = g.window > 0 ? pl.q_pos0 + 1 - g.window : 0;
  int64_t tq = 0, touched = 0;
  for (int64_t grp = pl.g_first; grp < pl.st.n_groups; ++grp) {
    const int64_t a0 = g.S + grp * g.G, a1 = a0 + g.G;
    const int64_t start = a0 > lo ? a0 : lo;
    const int64_t vis = a1 - start;
    if (vis > 0) { tq += vis; touched += 1; }
  }
  const int64_t per_unit = 2 * tq * d * g.bits / 8 + 4 * d * touched + 4 * tq + 4 * d * pl.st.n_res +
                           8 * d * pl.st.n_sink +
                           (g.n_out ? 2 * (2 * (g.G + 1) + 4 * static_cast<int64_t>(g.n_out)) * touched : 0);
  return per_unit * r.nb * g.hkv + 4 * d * static_cast<int64_t>(r.nb) * nq * g.hq;
}

// Query tokens per prefill call: bounded so that the units and the row
// indices stay well inside 32-bit kernel arithmetic.
constexpr int64_t kMaxQueries = 65536;
int64_t prefill_units(const Geo& g, int64_t nq) {
  return static_cast<int64_t>(g.B) * g.hkv * ((nq * g.rep + 3) / 4);
}
bool prefill_count_ok(const Geo& g, int64_t nq) {
  return nq >= 1 && nq <= kMaxQueries && prefill_units(g, nq) <= (int64_t{1} << 28);
}
// Scratch of a prefill call: [merge counters, one word per unit][partials,
// B * nq * h_q * split_stride records of d + 4 floats].
int64_t prefill_head_bytes(const Geo& g, int64_t nq) { return round_up(prefill_units(g, nq) * 4, kAlign); }
int64_t prefill_scratch_of(const Geo& g, int64_t nq) {
  return prefill_head_bytes(g, nq) +
         static_cast<int64_t>(g.B) * nq * g.hq * g.split_stride * (g.d + 4) * 4;
}

// The prefill attention over the runs of equal (T, n) with n = that run's
// query count (runs with none are skipped); q and out rows m_max per sequence.
int prefill_runs(kivi_cache* c, const std::vector<Run>& runs, const void* q, void* out, int64_t m_max,
                 void* scratch, cudaStream_t s) {
  const Geo& g = c->g;
  uint8_t* bytes = static_cast<uint8_t*>(scratch);
  const int64_t head = prefill_head_bytes(g, m_max);
  // the counters start at zero; every launch leaves them zero
  if (cudaMemsetAsync(bytes, 0, static_cast<size_t>(head), s) != cudaSuccess) return KIVI_ECUDA;
  for (const Run& r : runs) {
    if (r.n == 0) continue;
    const kivi::DecodePlan pl = plan_for(*c, r.T, r.nb, static_cast<int32_t>(r.n), static_cast<int32_t>(m_max));
    const cudaError_t e = attn_run(*c, r, pl, static_cast<const __half*>(q), static_cast<__half*>(out),
                                   reinterpret_cast<float*>(bytes + head), g.split_stride,
                                   reinterpret_cast<unsigned*>(bytes), ws_error(*c), s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KIVI_OK;
}
}  // namespace

int64_t kivi_decode_bytes(const kivi_cache* c) {
  if (!c) return -1;
  int64_t sum = 0;
  for (const Run& r : runs_of(*c)) sum += attn_bytes(*c, r, 1);
  return sum;
}

int64_t kivi_prefill_bytes(const kivi_cache* c, int64_t n_queries) {
  if (!c || n_queries > min_tokens_of(*c) || !prefill_count_ok(c->g, n_queries)) return -1;
  int64_t sum = 0;
  for (const Run& r : runs_of(*c)) sum += attn_bytes(*c, r, n_queries);
  return sum;
}

size_t kivi_prefill_scratch_bytes(const kivi_cache* c, int64_t n_queries) {
  if (!c || !prefill_count_ok(c->g, n_queries)) return 0;
  return static_cast<size_t>(prefill_scratch_of(c->g, n_queries));
}

int kivi_prefill_attn(kivi_cache* c, const void* q, void* out, int64_t n_queries, void* scratch,
                      size_t scratch_bytes, void* cuda_stream) {
  if (!c || !q || !out || !scratch) return KIVI_ENULL;
  if (n_queries > min_tokens_of(*c) || !prefill_count_ok(c->g, n_queries)) return KIVI_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(scratch, kAlign)) return KIVI_EALIGN;
  if (static_cast<int64_t>(scratch_bytes) < prefill_scratch_of(c->g, n_queries)) return KIVI_ENOSPC;
  return prefill_runs(c, runs_of(*c, [&](int32_t) { return n_queries; }), q, out, n_queries, scratch,
                      static_cast<cudaStream_t>(cuda_stream));
}

int kivi_prefill_attn_ragged(kivi_cache* c, const void* q, void* out, const int64_t* n_queries, int64_t m_max,
                             void* scratch, size_t scratch_bytes, void* cuda_stream) {
  if (!c || !q || !out || !scratch || !n_queries) return KIVI_ENULL;
  if (!prefill_count_ok(c->g, m_max)) return KIVI_EINVAL;
  for (int32_t b = 0; b < c->g.B; ++b)
    if (n_queries[b] < 0 || n_queries[b] > m_max || n_queries[b] > c->T[b]) return KIVI_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(scratch, kAlign)) return KIVI_EALIGN;
  if (static_cast<int64_t>(scratch_bytes) < prefill_scratch_of(c->g, m_max)) return KIVI_ENOSPC;
  return prefill_runs(c, runs_of(*c, [&](int32_t b) { return n_queries[b]; }), q, out, m_max, scratch,
                      static_cast<cudaStream_t>(cuda_stream));
}

int kivi_read_error(kivi_cache* c, uint32_t* flags, void* cuda_stream) {
  if (!c || !flags) return KIVI_ENULL;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  uint32_t word = 0;
  void* dev = c->arena + c->g.ws_error;
  if (cudaMemcpyAsync(&word, dev, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return KIVI_ECUDA;
  if (cudaMemsetAsync(dev, 0, 4, s) != cudaSuccess) return KIVI_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KIVI_ECUDA;
  *flags = word;
  return KIVI_OK;
}

const char* kivi_status_string(int status) {
  switch (status) {
    case KIVI_OK: return "ok";
    case KIVI_EINVAL: return "invalid parameter";
    case KIVI_EALIGN: return "pointer not aligned (arena: 256 bytes; tensors: 16 bytes)";
    case KIVI_ECAPACITY: return "append would exceed max_tokens";
    case KIVI_ENOSPC: return "arena smaller than kivi_cache_bytes()";
    case KIVI_ECUDA: return "CUDA launch or copy failed";
    case KIVI_ENULL: return "NULL pointer";
    case KIVI_ESCRATCH: return "problem too large for the library's fixed no-allocation scratch (4 MiB)";
    default: return "unknown status";
  }
}

}  // extern "C"
