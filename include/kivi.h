/*
 * kivi.h — C ABI of the GB300 (sm_103a) KIVI quantized KV cache.
 *
 * One library, libkivi.so, built from kivi_quantized_kv_gb300/csrc.  Plain
 * pointers and sizes only; no C++ or framework types cross this boundary and no
 * exception leaves it.
 *
 * What the cache computes (sources are the pages the method is described on):
 *   - KV-cache quantization guide (pigeon), "How it works", steps 1-5: keys
 *     quantized per channel with one scale and zero point per channel over a
 *     group of G tokens, values per token, asymmetric
 *     q = round((x - min) / Δ) with Δ = (max - min) / (2^b - 1); the most
 *     recent R tokens stay in fp16 until a group fills; decode attention
 *     softmax(q Kᵀ / sqrt(d)) V reads the packed groups and dequantizes them
 *     on the fly, never materialising an fp16 copy.
 *   - tract #2458 "quantized KV-cache storage op (int8/int4)": the first S
 *     tokens (attention sinks) stay in f32 in both stores; key blocks keep
 *     frozen scales once written.
 *   - tract #2329 "KIVI-style KV-cache quantization", "What's in the PR": a
 *     fused op over the query and the new keys and values, with grouped-query
 *     heads and an output shaped like the query; "Relationship to other PRs":
 *     a bounded sliding window composes with the quantized storage.
 *
 * Memory ownership: the caller allocates every device buffer (the arena,
 * prefill scratch and all inputs/outputs).  The library allocates only the
 * small host-side handle and never allocates or frees device memory; only
 * kivi_read_error synchronises a stream.
 *
 * Concurrency: every call is asynchronous on the given CUDA stream (NULL =
 * the legacy default stream).  A handle must not be used from two streams or
 * two host threads at the same time.
 *
 * Errors: each call returns a kivi_status.  All parameter checks run on the
 * host before any launch, so a call that returns an error has changed no
 * device or host state (except KIVI_ECUDA, raised when a launch itself
 * fails; the handle's token count is then left at its pre-call value).
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kivi_status {
  KIVI_OK = 0,
  KIVI_EINVAL = 1,     /* a parameter is outside the supported set */
  KIVI_EALIGN = 2,     /* a pointer is not aligned as required */
  KIVI_ECAPACITY = 3,  /* T + n would exceed max_tokens (window == 0) */
  KIVI_ENOSPC = 4,     /* the arena is smaller than kivi_cache_bytes() */
  KIVI_ECUDA = 5,      /* a CUDA launch or copy reported an error */
  KIVI_ENULL = 6,      /* a required pointer is NULL */
  KIVI_ESCRATCH = 7    /* too large for the fixed scratch of kivi_decode_attn_noalloc */
} kivi_status;

/* Cache parameters.
 *   bits       b in 1..8: code width (tract #2329: configurable width;
 *              kvquant++ README: 3 bits recommended).  b in {2, 4, 8} pack
 *              by the word rule below; the other widths pack as a bit
 *              stream and need G in {32, 64}.  Every width decodes on
 *              tensor cores at head dims 64 and 128.
 *   group      G: tokens per frozen key group; a multiple of 16 in [16, 256].
 *   residual   R: capacity of the fp16 residual ring; R >= G and R % G == 0.
 *   sinks      S in [0, 1024]: leading tokens kept in fp32.
 *   h_q, h_kv  query and key/value heads; h_q % h_kv == 0; query head h reads
 *              kv head h / (h_q / h_kv) (contiguous GQA groups).
 *   head_dim   d in {64, 128}.
 *   batch      B >= 1 sequences; each keeps its own token count (they grow
 *              alike through kivi_append and differently through
 *              kivi_append_ragged).
 *   max_tokens capacity in tokens per sequence when window == 0.
 *   window     W: 0 = attend to every token; W > 0 (W >= R) = attend to the
 *              sinks and to the most recent W tokens, the stream is unbounded
 *              and frozen groups live in a ring of ceil(W/G) + 1 slots. */
typedef struct kivi_params {
  int32_t bits;
  int32_t group;
  int32_t residual;
  int32_t sinks;
  int32_t h_q;
  int32_t h_kv;
  int32_t head_dim;
  int32_t batch;
  int64_t max_tokens;
  int64_t window;
  int32_t outlier_permille;   /* dense-and-sparse outliers: 0 = none, else
                                 1..50 per mille of each frozen key block and
                                 value block kept exactly (see the layout
                                 below); needs bits 2..4 and group a multiple
                                 of 32.  Decode, the fused step and the
                                 multi-query attention add the corrections */
  int32_t reserved;           /* 0 */
  double rope_base;           /* 0: keys arrive rotated (post-RoPE, or no
                                 RoPE).  > 1 (at most 1e7): pre-RoPE keys
                                 (KV-cache quantization guide (pigeon),
                                 "KVQuant adds"): keys are stored and
                                 quantized as they arrive, before the rotary
                                 embedding, and attention rotates each
                                 dequantized key at its own position a:
                                 channels (i, i + d/2) by the angle
                                 a * rope_base^(-2i/d); q arrives rotated.
                                 Needs group 32 or 64 and no outlier tables.
                                 Decode, the fused step and the multi-query
                                 attention run on tensor cores: the query is
                                 turned back by each group's first position
                                 and the keys by their offset inside the
                                 group (a table the handle writes once into
                                 the workspace) */
} kivi_params;

/* Byte layout of the arena and current state (all offsets in bytes).
 *
 * The arena is [cache region][workspace].  The cache region is B * h_kv
 * units, unit (b, h) at (b * h_kv + h) * unit_bytes; inside a unit:
 *   sink_k, sink_v  fp32 [S][d]        the sink tokens' keys / values
 *   res_k, res_v    fp16 [R][d]        ring; token a (>= S) in slot (a-S) % R
 *   groups          n_slots blocks of block_bytes; frozen group g (tokens
 *                   S+gG .. S+gG+G-1) in slot g (window == 0) or
 *                   g % n_slots (window > 0).  Inside a block:
 *     blk_kq  key codes, token-major: G rows of d*b/8 bytes
 *     blk_ks  fp16 key Δ[d] then key min[d] (one pair per channel)
 *     blk_vq  value codes, channel-major: d rows of G*b/8 bytes
 *     blk_vs  fp16 (Δ, min) per token, G pairs
 *     blk_ko, blk_vo  (outlier_permille > 0) key and value outlier tables,
 *             rows by token: u16 row pointers [G + 1] (the entries of
 *             token t are [ptr[t], ptr[t+1])), then from out_entries the
 *             n_outliers = ceil(outlier_permille * G * d / 1000) entries
 *             of 4 bytes {u8 token t, u8 channel c, fp16 value}, in
 *             increasing t * d + c; each table padded to 16 bytes.  The
 *             outliers of a block are its n_outliers values of largest
 *             magnitude (ties to the smaller t * d + c); they are left out
 *             of the dense min and max, take code 0 and read back exactly
 *             (KV-cache quantization guide (pigeon), "KVQuant adds": a
 *             small share of values kept in fp16 beside the codes).
 *   b in {2, 4, 8}: a row of codes is cut into little-endian 32-bit words
 *   of 32/b codes; element j of a word sits in the low 16-bit half when j is
 *   even, the high half when j is odd, at bit b*floor(j/2) of its half.
 *   Other b: a bit stream, element j at bits [b j, b j + b) of the row from
 *   the least significant bit of byte 0 (codes cross byte boundaries).
 * The workspace (workspace_offset, workspace_bytes) holds split-K partial
 * results and per-unit counters; its contents are scratch. */
typedef struct kivi_layout {
  int64_t n_slots;
  int64_t sink_k, sink_v, res_k, res_v, groups;
  int64_t block_bytes, blk_kq, blk_ks, blk_vq, blk_vs;
  int64_t unit_bytes, cache_bytes;
  int64_t workspace_offset, workspace_bytes, arena_bytes;
  int64_t tokens;     /* T: tokens appended per sequence; -1 when the
                         sequences' counts differ (kivi_cache_tokens);
                         the three fields below are sequence 0's */
  int64_t n_sink;     /* min(T, S) */
  int64_t n_groups;   /* frozen groups written so far */
  int64_t n_res;      /* tokens live in the ring */
  int32_t max_splits; /* CTAs that may share one unit's work */
  int32_t reserved;
  int64_t blk_ko, blk_vo;   /* outlier tables inside a block */
  int64_t n_outliers;       /* entries per table (0 without outliers) */
  int64_t out_entries;      /* offset of the entries inside a table */
} kivi_layout;

typedef struct kivi_cache kivi_cache;

/* Bytes of device memory the arena needs (cache region + workspace), or 0 if
 * the parameters are invalid.  Host only; touches no device. */
size_t kivi_cache_bytes(const kivi_params* params);

/* Creates a handle over a caller-owned device arena of at least
 * kivi_cache_bytes(params) bytes, 256-byte aligned, and zeroes the arena
 * asynchronously on `stream`.  *out receives the handle (host memory owned by
 * the library until kivi_cache_destroy).  Errors: ENULL, EINVAL, EALIGN,
 * ENOSPC, ECUDA. */
int kivi_cache_create(const kivi_params* params, void* d_arena, size_t arena_bytes,
                      void* cuda_stream, kivi_cache** out);

/* Re-attaches a handle to an arena that already holds a cache written by this
 * library with the same parameters (checkpoint / resume: the arena's cache
 * region, the kivi_params and the B token counts are the whole state, so a
 * byte copy of the arena taken after its stream was synchronised, with
 * kivi_cache_tokens, restores it; no file format).  tokens: host array of B
 * counts.  Unlike kivi_cache_create it keeps the cache region; it clears the
 * workspace's merge counters and error word on `stream`.  Errors: ENULL,
 * EINVAL (parameters, or a count < 0, or above max_tokens when window == 0),
 * EALIGN, ENOSPC, ECUDA. */
int kivi_cache_restore(const kivi_params* params, void* d_arena, size_t arena_bytes, const int64_t* tokens,
                       void* cuda_stream, kivi_cache** out);

/* Host-side fault injection for tests of the error paths (the method's pages
 * have no counterpart): n >= 1 arms the n-th kernel launch the library makes
 * from now on, in any handle of the process, to fail with ECUDA without
 * being made; the call that hits it returns ECUDA with its token counts
 * unchanged (launches it made before stay made).  0 disarms.  Nothing is
 * injected on the device.  Errors: EINVAL (n < 0). */
int kivi_debug_inject_launch_failure(int64_t n);

/* Host-side control of the decode's bounded copy waits, for tests of the
 * error path (the method's pages have no counterpart).  Every decode warp
 * waits at most this long for each of its copies into shared memory; when a
 * wait runs out the warp stops consuming, lets the copies it issued land
 * (those waits keep the 2 s bound), and sets bit 0 of the cache's error word
 * (kivi_read_error), so the call's outputs are invalid but the launch ends.
 * ns >= 1 sets the limit for launches made from now on, in any handle of
 * the process; 0 restores the default of 2 s.  A limit of a few nanoseconds
 * makes waits run out while the copies are still in flight.
 * Errors: EINVAL (ns < 0). */
int kivi_debug_set_wait_limit(int64_t ns);

/* Frees the host handle.  The arena stays the caller's. */
void kivi_cache_destroy(kivi_cache* cache);

/* Appends n_tokens (>= 1) new tokens to every sequence (KV-cache
 * quantization guide, steps 1-4; tract #2458 sinks).
 *   k_new, v_new  device fp16 [B][h_kv][n_tokens][d], contiguous, 16-byte
 *                 aligned.
 * Tokens below position S are widened to fp32 sink slots.  A token that
 * reaches a full ring first pushes the ring's oldest G tokens out as one
 * frozen group: keys quantized per channel over the G tokens, values per
 * token, codes packed and (Δ, min) stored as fp16.  The ring then receives
 * the token.  Bulk appends give the same bytes as token-by-token appends.
 * Errors: ENULL, EALIGN, EINVAL (n_tokens < 1), ECAPACITY, ECUDA. */
int kivi_append(kivi_cache* cache, const void* k_new, const void* v_new, int64_t n_tokens,
                void* cuda_stream);

/* Appends a different number of tokens to each sequence (ragged batches:
 * chunked prefill of sequences of different lengths).
 *   k_new, v_new  device fp16 [B][h_kv][n_max][d], contiguous, 16-byte
 *                 aligned; row (b, h) holds sequence b's new tokens first,
 *                 the rest of the row is ignored.
 *   n_tokens      host array of B counts, each in [0, n_max].
 * Each sequence's bytes are those kivi_append would give it alone.  The
 * library launches the append once per run of consecutive sequences with
 * equal (length, count).  Errors: ENULL, EALIGN, EINVAL (n_max < 1 or a
 * count outside [0, n_max]), ECAPACITY, ECUDA. */
int kivi_append_ragged(kivi_cache* cache, const void* k_new, const void* v_new, const int64_t* n_tokens,
                       int64_t n_max, void* cuda_stream);

/* Token counts of the B sequences into the host array tokens[B].
 * Errors: ENULL. */
int kivi_cache_tokens(const kivi_cache* cache, int64_t* tokens);

/* Decode attention over everything appended so far (KV-cache quantization
 * guide, step 5; tract #2329 GQA and output shape).
 *   q    device fp16 [B][h_q][d], contiguous, 16-byte aligned.
 *   out  device fp16 [B][h_q][d], contiguous, 16-byte aligned.
 * out[b][h] = Σ_t softmax_t(q·k̂_t / sqrt(d)) v̂_t over the visible tokens of
 * kv head h / (h_q / h_kv): the sinks (fp32), the frozen groups (dequantized
 * in registers) and the ring (fp16); with a window, the sinks plus the most
 * recent W tokens.  With T == 0 the output is all zeros.  The work is split
 * over the sequence (split-K) and merged in the same call; the workspace is
 * scratch.  Sequences of different lengths each attend over their own
 * tokens: the batch is cut into runs of consecutive sequences of equal
 * length and one launch covers up to 64 runs (the runs' plans travel in the
 * launch's parameters), so a ragged batch of up to 64 distinct lengths is
 * still one launch.  Errors: ENULL, EALIGN, ECUDA. */
int kivi_decode_attn(kivi_cache* cache, const void* q, void* out, void* cuda_stream);

/* One decode step in one call: appends one token to every sequence and
 * returns the decode attention over everything including that token, the
 * fused op of tract #2329, "What's in the PR" (it takes the query with the
 * new keys and values and returns an output shaped like the query).  The result and the cache bytes are those of
 * kivi_append(k_new, v_new, 1) followed by kivi_decode_attn(q, out) (the
 * output to within the decode's rounding).  The new token is attended
 * straight from k_new / v_new and written into its sink or ring slot by the
 * decode launch itself, so a step is one launch; a step whose token freezes
 * a group (the ring is full) first runs that group's quantization launch.
 * Sequences of different lengths: as kivi_decode_attn, one decode launch per
 * 64 runs, preceded by one quantization launch over the sequences whose
 * token freezes a group.
 *   k_new, v_new  device fp16 [B][h_kv][1][d], contiguous, 16-byte aligned.
 *   q, out        device fp16 [B][h_q][d], contiguous, 16-byte aligned.
 * Errors: ENULL, EALIGN, ECAPACITY, ECUDA (the token count is then left
 * at its pre-call value). */
int kivi_append_decode_attn(kivi_cache* cache, const void* k_new, const void* v_new, const void* q, void* out,
                            void* cuda_stream);

/* Same as kivi_append_decode_attn with host-resident k_new, v_new, q and out.
 * When all four are pinned host memory mapped into the device's address
 * space (cudaHostAlloc / cudaMallocHost / cudaHostRegister under unified
 * addressing) and 16-byte aligned, the step reads the inputs over that
 * mapping and writes its output straight to out_host (no copy engine
 * involved; for bit-stream widths, outlier tables and pre-RoPE keys one extra
 * launch first gathers the inputs into the arena's staging area); otherwise
 * (pageable memory) the call copies the inputs into the staging area, runs
 * the step and copies the result back to out_host.  Everything is queued on `stream`, in stream
 * order.  Either way the call returns once the work is
 * queued: synchronise the stream before reading out_host or reusing the input
 * buffers.  Errors: as kivi_append_decode_attn. */
int kivi_append_decode_attn_host(kivi_cache* cache, const void* k_host, const void* v_host, const void* q_host,
                                 void* out_host, void* cuda_stream);

/* Same as kivi_decode_attn with host-resident q and out: a pinned, mapped,
 * 16-byte aligned q is read over the mapping and the output written straight
 * to out_host; other memory is staged through the arena with copies on
 * `stream` (as kivi_append_decode_attn_host).  The call returns once the work is
 * queued; synchronise the stream before reading out_host.  Errors: as
 * kivi_decode_attn. */
int kivi_decode_attn_host(kivi_cache* cache, const void* q_host, void* out_host, void* cuda_stream);

/* Causal attention of the n_queries newest tokens of every sequence over the
 * cache (chunked prefill: kvquant++ README, long-document example, where
 * prefill_chunk_size bounds each attention step to one chunk of queries while
 * the context accumulates in the cache; the per-query attention is that of
 * kivi_decode_attn).  Append the chunk first (kivi_append), then call this
 * with the chunk's queries.
 *   q    device fp16 [B][n_queries][h_q][d], contiguous, 16-byte aligned;
 *        query j of a sequence is the token at position T - n_queries + j.
 *   out  device fp16 [B][n_queries][h_q][d], contiguous, 16-byte aligned.
 *   scratch  device memory of at least kivi_prefill_scratch_bytes(cache,
 *        n_queries) bytes, 256-byte aligned, owned by the caller; its
 *        contents are scratch (the call clears what it needs on `stream`).
 * Query j attends to the tokens at positions <= T - n_queries + j that the
 * cache holds: the sinks (fp32), frozen groups (dequantized in registers) and
 * the ring (fp16), as the cache stands after the append (a chunk token that
 * the append froze is read from its codes); with a window, the sinks plus the
 * W tokens ending at the query's own position, less any whose group slot the
 * window's ring has reused (a chunk longer than about R tokens can lose the
 * oldest part of its first queries' windows).  The newest query's row equals
 * kivi_decode_attn's output for it.  Work: as kivi_decode_attn with n_queries
 * times the query rows per kv head, each row masked to its own positions.
 * Errors: ENULL, EINVAL (n_queries < 1, > T or > 65536), EALIGN, ENOSPC
 * (scratch too small), ECUDA. */
int kivi_prefill_attn(kivi_cache* cache, const void* q, void* out, int64_t n_queries, void* scratch,
                      size_t scratch_bytes, void* cuda_stream);

/* kivi_prefill_attn for sequences of different lengths and chunk sizes:
 * sequence b's n_queries[b] newest tokens attend, each to the tokens at or
 * before its own position in that sequence (n_queries: host array of B
 * counts in [0, min(m_max, its token count)]).
 *   q, out  device fp16 [B][m_max][h_q][d]; rows j >= n_queries[b] of a
 *           sequence are not read (q) and not written (out).
 *   scratch at least kivi_prefill_scratch_bytes(cache, m_max) bytes.
 * One launch per run of consecutive sequences with equal (length, count).
 * Errors: ENULL, EINVAL (as kivi_prefill_attn), EALIGN, ENOSPC, ECUDA. */
int kivi_prefill_attn_ragged(kivi_cache* cache, const void* q, void* out, const int64_t* n_queries,
                             int64_t m_max, void* scratch, size_t scratch_bytes, void* cuda_stream);

/* Device scratch bytes kivi_prefill_attn needs for n_queries query tokens per
 * sequence (independent of T), or 0 for a NULL handle or an n_queries outside
 * [1, 65536].  Host only. */
size_t kivi_prefill_scratch_bytes(const kivi_cache* cache, int64_t n_queries);

/* Algorithmic bytes of one kivi_prefill_attn call at the current state: the
 * cache bytes of every token some query sees (as kivi_decode_bytes counts
 * them) plus q and out.  -1 for a NULL handle or an invalid n_queries. */
int64_t kivi_prefill_bytes(const kivi_cache* cache, int64_t n_queries);

/* Reads and clears the device error word that the cache's attention launches
 * (kivi_decode_attn, kivi_append_decode_attn, kivi_prefill_attn and
 * kivi_decode_attn_noalloc, with their variants) set instead of hanging:
 * bit 0 = a bulk copy into shared memory did not complete within its bounded
 * wait (2 s, or the limit of kivi_debug_set_wait_limit), bit 1 = a warp
 * waited in vain for its combine slot to be released.  Either bit means the
 * affected outputs are not valid.  The checked build of the library
 * (libkivi_debug.so, compiled with KIVI_DEBUG_CHECKS=1) adds two bits that
 * every kernel, appends included, may set: bit 2 = an arena address derived
 * from the plan left the cache region (the access was skipped), bit 3 = an
 * input key, value or query element was inf or NaN (a precondition of the
 * method; the product build does not look).  Unlike every other call this
 * one synchronises `stream` (it returns the value).  Errors: ENULL, ECUDA. */
int kivi_read_error(kivi_cache* cache, uint32_t* flags, void* cuda_stream);

/* Decode attention that allocates nothing (the method's pages have no
 * counterpart: this is a deployment variant of kivi_decode_attn).  For callers
 * that can pass only their inputs and outputs and cannot obtain device memory
 * while decoding, for instance a plugin inside a host runtime that owns all
 * device memory and forbids allocation during execution.  Same arguments,
 * layouts and result as kivi_decode_attn (within its rounding: the split
 * count may be lower); the split-K scratch is a fixed 4 MiB device array
 * inside the library instead of the arena workspace.  It calls no cudaMalloc
 * or cudaFree.
 *   - Every GPU that loads the library holds the 4 MiB until process exit;
 *     the CUDA driver materialises it when it loads the library's device
 *     variables (with lazy module loading, at the latest on the first call).
 *   - The first call on a device looks up the array's device address on the
 *     current device; make that first call before any stream capture.
 *   - All calls share the array: calls whose GPU work overlaps (concurrent
 *     streams or host threads) race on it.  The merge counters in it are
 *     cleared by every call.
 *   - The bounded waits report into the cache's own error word, which lives
 *     in the arena the caller already owns: read it with kivi_read_error.
 *   - Three partial records per query head, 3 * B * h_q * (head_dim + 4) * 4
 *     bytes, plus the merge counters must fit in 4 MiB, else KIVI_ESCRATCH and
 *     nothing runs; the work is spread over fewer CTAs when fewer records fit.
 * Errors: ENULL, EALIGN, ESCRATCH, ECUDA. */
int kivi_decode_attn_noalloc(kivi_cache* cache, const void* q, void* out, void* cuda_stream);

/* Forces the number of CTAs per (sequence, kv head) unit that later decode
 * calls spread the work over (0 = the library's own choice: one wave of
 * resident CTAs; larger values are clamped to what the workspace holds).
 * Errors: ENULL, EINVAL (negative). */
int kivi_set_num_splits(kivi_cache* cache, int32_t num_splits);

/* Layout, counters and sizes of the handle.  Errors: ENULL. */
int kivi_cache_layout(const kivi_cache* cache, kivi_layout* out);

/* The layout a cache of these parameters has, without creating one (host
 * only; touches no device): every offset and size as kivi_cache_layout
 * reports it, the state fields those of an empty cache (tokens 0).
 * Errors: ENULL, EINVAL (invalid parameters). */
int kivi_layout_for(const kivi_params* params, kivi_layout* out);

/* Algorithmic bytes one decode call must move at the current state: packed
 * codes of the visible quantized tokens, key (Δ, min) rows of the groups they
 * touch, value (Δ, min) pairs, fp16 ring tokens, fp32 sinks, q and out.
 * Returns -1 for a NULL handle. */
int64_t kivi_decode_bytes(const kivi_cache* cache);

/* Static text for a status code. */
const char* kivi_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_H */
