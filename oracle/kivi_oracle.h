/*
 * kivi_oracle.h — plain, slow CPU oracle for the KIVI quantized KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * in __graft_entry__.py and the CPU-baseline leg of bench.py may load this
 * library.  It shares no code, header, table or helper with the CUDA library
 * under kivi_quantized_kv_gb300/; neither side includes or links the other.
 *
 * What it computes (sources are the pages the method is described on):
 *   - KV-cache quantization guide (pigeon), "How it works", steps 1-5:
 *       keys per channel over groups of G tokens, values per token,
 *       asymmetric q = round((x - min) / Δ), Δ = (max - min) / (2^b - 1),
 *       full-precision residual window of the most recent R tokens,
 *       softmax(q Kᵀ / sqrt(d)) V over the dequantized values.
 *   - tract #2458 "quantized KV-cache storage op (int8/int4)", commit on
 *       attention sinks: the first SINK tokens are kept in f32 in both stores.
 *   - tract #2458 description: keys quantized in fixed-size blocks whose
 *       scales never change once written, so a stream gives the same bytes
 *       however it is chunked.
 *   - tract #2329 "KIVI-style KV-cache quantization", "What's in the PR":
 *       grouped-query heads; the op takes the query with the new keys and
 *       values, and its output is shaped like the query.
 *   - tract #2329 "Relationship to other PRs": bounded sliding-window cache
 *       composed with quantization.
 *
 * All fp16 values cross this interface as their IEEE binary16 bit patterns
 * (uint16_t).  Status codes match the CUDA library's meaning (0 = OK,
 * 1 = invalid parameter, 3 = capacity exceeded).
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ko_params {
  int32_t bits;      /* b in 1..8 (2, 4, 8: word rule; others: bit stream) */
  int32_t group;     /* G: tokens per frozen key group */
  int32_t residual;  /* R: capacity of the fp16 residual ring */
  int32_t sinks;     /* S: leading tokens kept in fp32 */
  int32_t h_q;       /* query heads */
  int32_t h_kv;      /* key/value heads */
  int32_t head_dim;  /* d */
  int32_t batch;     /* B */
  int64_t max_tokens;/* capacity T_max when window == 0 */
  int64_t window;    /* W: 0 = attend to everything; > 0 = sinks + last W tokens */
  int32_t outlier_permille; /* dense-and-sparse: per frozen key block and value
                               block, ceil(permille * G * d / 1000) values kept
                               exactly in a side table; 0 = none */
  int32_t window_mode; /* the two readings of a window composed with sinks
                          (tract #2329 "Relationship to other PRs" gives no
                          sink rule): 0 = the sinks stay visible beside the
                          most recent W tokens (the CUDA library's reading);
                          1 = a pure window, the sinks expire like any other
                          token once they leave the most recent W */
  double rope_base;  /* 0: keys arrive rotated (post-RoPE).  > 1: keys arrive
                        and are stored before RoPE; attention rotates each
                        dequantized key at its position (rotate-half pairs
                        (i, i + d/2), angle position * base^(-2i/d)) */
} ko_params;

/* Byte layout of one (batch, kv-head) unit and of one frozen group block. */
typedef struct ko_layout {
  int64_t n_slots;        /* frozen-group slots per unit */
  int64_t sink_k, sink_v; /* offsets inside a unit: fp32 [S][d] each */
  int64_t res_k, res_v;   /* fp16 [R][d] each */
  int64_t groups;         /* first group block */
  int64_t block_bytes;    /* one group block */
  int64_t blk_kq, blk_ks, blk_vq, blk_vs; /* offsets inside a block */
  int64_t blk_ko, blk_vo; /* key and value outlier tables (CSR by token):
                             u16 row pointers [G + 1], then, from
                             out_entries, n_outliers entries of
                             {u8 token, u8 channel, fp16 value} */
  int64_t n_outliers;     /* entries per table (0 without outliers) */
  int64_t out_entries;    /* offset of the entries inside a table */
  int64_t unit_bytes;     /* one (b, h_kv) unit */
  int64_t cache_bytes;    /* B * H_kv * unit_bytes */
} ko_layout;

/* ---- IEEE binary16 conversion (written from the format definition) ---- */
uint16_t ko_f32_to_f16(float x);                 /* round to nearest, ties to even */
float ko_f16_to_f32(uint16_t h);                 /* exact */
void ko_f32_to_f16_array(const float* x, uint16_t* out, int64_t n);
void ko_f16_to_f32_array(const uint16_t* h, float* out, int64_t n);

/* ---- one asymmetric quantization of n values (x[i*stride]) ----
 * Writes n codes (one per byte, unpacked) and the fp16 (Δ, min) pair. */
void ko_quantize(const uint16_t* x, int32_t n, int64_t stride, int32_t bits,
                 uint8_t* codes, uint16_t* delta16, uint16_t* min16);

/* ---- packing of one row of L codes into L*bits/8 bytes, and its inverse ---- */
int ko_pack_row(const uint8_t* codes, int32_t L, int32_t bits, uint8_t* out);
int ko_unpack_row(const uint8_t* packed, int32_t L, int32_t bits, uint8_t* codes);

/* ---- cache ---- */
int ko_validate(const ko_params* p);
int ko_layout_of(const ko_params* p, ko_layout* out);
/* State counters as a pure function of the token count T. */
void ko_state_of(const ko_params* p, int64_t T, int64_t* n_sink, int64_t* n_groups, int64_t* n_res);

typedef struct ko_cache ko_cache;
int ko_create(const ko_params* p, ko_cache** out);
void ko_destroy(ko_cache* c);
/* Appends n tokens per (batch, kv-head): k_new, v_new are [B][H_kv][n][d] fp16. */
int ko_append(ko_cache* c, const uint16_t* k_new, const uint16_t* v_new, int64_t n);
int64_t ko_tokens(const ko_cache* c);
int64_t ko_groups(const ko_cache* c);
int64_t ko_residual_count(const ko_cache* c);
const uint8_t* ko_arena(const ko_cache* c);

/* Decoded view of one unit: K̂, V̂ [T][d] (fp64) and a visibility flag per token. */
int ko_dequant_unit(const ko_cache* c, int32_t b, int32_t hkv, double* k_hat, double* v_hat,
                    uint8_t* visible);

/* Decode attention, fp64: q [B][H_q][d] fp16 -> out [B][H_q][d] fp64.
 * Work is spread over `threads` host threads by (batch, kv-head) unit. */
int ko_decode_attn(const ko_cache* c, const uint16_t* q, double* out, int32_t threads);

/* Causal attention of the n_queries newest tokens, fp64: q [B][M][H_q][d]
 * fp16 -> out [B][M][H_q][d] fp64, query j at position T - M + j attending to
 * the resident tokens a <= T - M + j (sinks, and with a window the W tokens
 * ending at its own position).  1 <= n_queries <= T, else 1 (invalid). */
int ko_prefill_attn(const ko_cache* c, const uint16_t* q, int64_t n_queries, double* out, int32_t threads);

/* Algorithmic bytes one decode pass must read/write at the current state. */
int64_t ko_decode_bytes(const ko_cache* c);

#ifdef __cplusplus
}
#endif
#endif
