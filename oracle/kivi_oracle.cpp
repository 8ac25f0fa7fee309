// kivi_oracle.cpp — plain, slow, obviously-correct CPU oracle for the KIVI
// quantized KV cache and decode attention.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, the smoke check and
// the CPU-baseline leg of the benchmark load it.  It shares no code with the
// CUDA library.  Build flags: -O2 -ffp-contract=off, no fast-math, so every
// fp32 operation below is one separately rounded IEEE operation.
//
// Every step follows the pages' order:
//   KV-cache quantization guide (pigeon), "How it works":
//     1. keys per channel, one scale and zero point per channel over a group
//        of G tokens;
//     2. values per token, one scale and zero point per token;
//     3. q = round((x - min) / Δ), Δ = (max - min) / (2^b - 1);
//     4. the most recent R tokens stay in fp16 and are quantized once a
//        group fills;
//     5. softmax(q Kᵀ / sqrt(d)) V over the dequantized values.
//   tract #2458 (quantized KV-cache storage op), sink commit: the first S
//     tokens stay in f32 in both the key and the value store.
//   tract #2458 description: key blocks have frozen scales.
//   tract #2329 "What's in the PR": GQA is handled (query heads share a KV
//     head).
// Readings where the pages are silent are stated beside the code that takes
// them.
#include "kivi_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kOk = 0;
constexpr int kInvalid = 1;
constexpr int kCapacity = 3;

// ---------------------------------------------------------------------------
// IEEE-754 binary16 <-> binary32, from the format definition:
// binary16 = 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
// subnormals have exponent field 0 and value fraction * 2^-24.
// ---------------------------------------------------------------------------
uint32_t bits_of(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float float_of(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// Right shift of a significand by `shift` bits with round-to-nearest, ties to
// even.  shift is in [1, 31].
uint32_t shift_round_even(uint32_t sig, int shift) {
  const uint32_t q = sig >> shift;
  const uint32_t rem = sig & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) return q + 1u;
  return q;
}

uint16_t f32_to_f16(float f) {
  const uint32_t x = bits_of(f);
  const uint16_t sign = static_cast<uint16_t>((x >> 16) & 0x8000u);
  const uint32_t exp = (x >> 23) & 0xFFu;
  const uint32_t frac = x & 0x7FFFFFu;
  if (exp == 0xFFu) {                      // infinity or NaN
    if (frac == 0) return sign | 0x7C00u;
    return sign | 0x7E00u;                 // a quiet NaN
  }
  if (exp == 0) return sign;               // fp32 zero/subnormal: far below 2^-25
  const int e = static_cast<int>(exp) - 127;   // unbiased exponent
  const uint32_t sig = frac | 0x800000u;       // 24-bit significand, value sig*2^(e-23)
  if (e >= -14) {                              // lands in the binary16 normal range
    uint32_t q = shift_round_even(sig, 13);    // 11-bit significand in [1024, 2048]
    int he = e + 15;
    if (q == 2048u) { q = 1024u; ++he; }
    if (he >= 31) return sign | 0x7C00u;       // overflow to infinity
    return static_cast<uint16_t>(sign | (he << 10) | (q & 0x3FFu));
  }
  // binary16 subnormal: count of 2^-24 units = sig * 2^(e+1)
  const int shift = -(e + 1);                  // >= 14
  if (shift > 24) return sign;                 // below half of 2^-24
  const uint32_t q = shift_round_even(sig, shift);   // may round up to 1024 = min normal
  return static_cast<uint16_t>(sign | q);
}

float f16_to_f32(uint16_t h) {
  const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1Fu;
  const uint32_t m = h & 0x3FFu;
  if (e == 0) {
    const float mag = std::ldexp(static_cast<float>(m), -24);   // exact
    return (sign != 0) ? -mag : mag;
  }
  if (e == 31) return float_of(sign | 0x7F800000u | (m << 13));
  return float_of(sign | ((e - 15 + 127) << 23) | (m << 13));
}

// ---------------------------------------------------------------------------
// Asymmetric quantizer (pigeon guide, "How it works", step 3):
//   q = round((x - min) / Δ),  Δ = (max - min) / (2^b - 1).
// Readings (the pages are silent on the arithmetic):
//   * x values are fp16 widened exactly to fp32; every operation is one
//     IEEE fp32 operation rounded to nearest-even, no fused multiply-add;
//   * min and max are canonicalised with + 0.0f so that -0 becomes +0;
//   * Δ and the zero point are stored as fp16, and the STORED fp16 Δ is the
//     divisor that makes the codes;
//   * "round" is round-half-to-even; codes are clamped to [0, 2^b - 1]
//     (the fp16 Δ can be a little smaller than the exact one);
//   * when the stored Δ is zero (a constant vector) every code is 0.
// The zero point is the fp16 min itself (exact, because min is an fp16 value).
// ---------------------------------------------------------------------------
// skip (may be null): elements kept exactly in an outlier table; they take
// no part in min and max and get code 0.  A vector whose every element is
// skipped gets min = 0, Δ = 0.
void quantize(const uint16_t* x, int n, int64_t stride, int bits, uint8_t* codes,
              uint16_t* d16_out, uint16_t* mn16_out, const uint8_t* skip = nullptr) {
  float mn = std::numeric_limits<float>::infinity();
  float mx = -std::numeric_limits<float>::infinity();
  for (int i = 0; i < n; ++i) {
    if (skip && skip[i * stride]) continue;
    const float v = f16_to_f32(x[i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  if (mn > mx) { mn = 0.0f; mx = 0.0f; }   // every element is an outlier
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  const int top = (1 << bits) - 1;
  const float delta = (mx - mn) / static_cast<float>(top);
  const uint16_t d16 = f32_to_f16(delta);
  const float dq = f16_to_f32(d16);
  for (int i = 0; i < n; ++i) {
    int code = 0;
    if (dq != 0.0f && !(skip && skip[i * stride])) {
      const float v = f16_to_f32(x[i * stride]);
      const float t = (v - mn) / dq;
      const float r = std::nearbyint(t);          // default mode: nearest, ties to even
      code = static_cast<int>(std::min(std::max(r, 0.0f), static_cast<float>(top)));
    }
    codes[i] = static_cast<uint8_t>(code);
  }
  *d16_out = d16;
  *mn16_out = f32_to_f16(mn);
}

// ---------------------------------------------------------------------------
// Packing of one row of L codes of b bits (the pages fix only "packed u8").
// Reading for b in {2, 4, 8}: the row is cut into little-endian 32-bit words
// of 32/b codes; in each word, row element j (0-based inside the word) sits
// in the low 16-bit half when j is even and in the high half when j is odd,
// at bit offset b * floor(j/2) inside its half, least significant first.
// Reading for the other widths (b in {1, 3, 5, 6, 7}; tract #2329 allows
// 1..16 bits, kvquant++ recommends 3): a plain bit stream, element j at bits
// [b j, b j + b) of the row counted from the least significant bit of byte 0,
// so codes cross byte boundaries and no bit is left empty.
// ---------------------------------------------------------------------------
bool word_rule(int bits) { return bits == 2 || bits == 4 || bits == 8; }

int pack_stream(const uint8_t* codes, int L, int bits, uint8_t* out) {
  if ((static_cast<int64_t>(L) * bits) % 8 != 0) return kInvalid;
  const int64_t nbytes = static_cast<int64_t>(L) * bits / 8;
  for (int64_t i = 0; i < nbytes; ++i) out[i] = 0;
  for (int j = 0; j < L; ++j) {
    for (int k = 0; k < bits; ++k) {
      const int64_t bit = static_cast<int64_t>(j) * bits + k;
      if ((codes[j] >> k) & 1) out[bit / 8] = static_cast<uint8_t>(out[bit / 8] | (1u << (bit % 8)));
    }
  }
  return kOk;
}

int unpack_stream(const uint8_t* packed, int L, int bits, uint8_t* codes) {
  if ((static_cast<int64_t>(L) * bits) % 8 != 0) return kInvalid;
  for (int j = 0; j < L; ++j) {
    int c = 0;
    for (int k = 0; k < bits; ++k) {
      const int64_t bit = static_cast<int64_t>(j) * bits + k;
      c |= ((packed[bit / 8] >> (bit % 8)) & 1) << k;
    }
    codes[j] = static_cast<uint8_t>(c);
  }
  return kOk;
}

int pack_row(const uint8_t* codes, int L, int bits, uint8_t* out) {
  if (!word_rule(bits)) return pack_stream(codes, L, bits, out);
  if ((static_cast<int64_t>(L) * bits) % 32 != 0) return kInvalid;
  const int per = 32 / bits;
  for (int w = 0; w < L / per; ++w) {
    uint32_t word = 0;
    for (int j = 0; j < per; ++j) {
      const uint32_t c = codes[w * per + j];
      const int shift = 16 * (j & 1) + bits * (j >> 1);
      word |= c << shift;
    }
    for (int k = 0; k < 4; ++k) out[4 * w + k] = static_cast<uint8_t>(word >> (8 * k));
  }
  return kOk;
}

int unpack_row(const uint8_t* packed, int L, int bits, uint8_t* codes) {
  if (!word_rule(bits)) return unpack_stream(packed, L, bits, codes);
  if ((static_cast<int64_t>(L) * bits) % 32 != 0) return kInvalid;
  const int per = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
  for (int w = 0; w < L / per; ++w) {
    uint32_t word = 0;
    for (int k = 0; k < 4; ++k) word |= static_cast<uint32_t>(packed[4 * w + k]) << (8 * k);
    for (int j = 0; j < per; ++j) {
      const int shift = 16 * (j & 1) + bits * (j >> 1);
      codes[w * per + j] = static_cast<uint8_t>((word >> shift) & mask);
    }
  }
  return kOk;
}

// ---------------------------------------------------------------------------
// Parameters, state and layout.
// ---------------------------------------------------------------------------
int validate(const ko_params& p) {
  if (p.bits < 1 || p.bits > 8) return kInvalid;   // codes are bytes here; wider codes are out of scope
  if (!(p.head_dim == 64 || p.head_dim == 128)) return kInvalid;
  if (p.group < 16 || p.group > 256 || p.group % 16 != 0) return kInvalid;
  if (p.residual < p.group || p.residual % p.group != 0) return kInvalid;
  if (p.sinks < 0 || p.sinks > 1024) return kInvalid;
  if (p.h_kv < 1 || p.h_q < 1 || p.h_q % p.h_kv != 0) return kInvalid;
  if (p.batch < 1) return kInvalid;
  if (p.window < 0 || p.max_tokens < 0) return kInvalid;
  if (p.window > 0 && p.window < p.residual) return kInvalid;
  if (p.outlier_permille < 0 || p.outlier_permille > 50) return kInvalid;
  if (p.window_mode != 0 && p.window_mode != 1) return kInvalid;
  if (!(p.rope_base == 0.0 || (p.rope_base > 1.0 && p.rope_base <= 1e7))) return kInvalid;
  return kOk;
}

// Frozen groups and residual tokens after T tokens (lazy flush reading of
// "keep the most recent R tokens in fp16 and quantize them once a group
// fills"): a token that arrives at a full ring first pushes the ring's oldest
// G tokens out as one frozen group.
void state_of(const ko_params& p, int64_t T, int64_t* n_sink, int64_t* n_groups, int64_t* n_res) {
  const int64_t S = p.sinks, R = p.residual, G = p.group;
  const int64_t ns = std::min<int64_t>(T, S);
  const int64_t m = std::max<int64_t>(T - S, 0);
  const int64_t ng = (m <= R) ? 0 : (m - R + G - 1) / G;
  *n_sink = ns;
  *n_groups = ng;
  *n_res = m - ng * G;
}

int64_t slots_of(const ko_params& p) {
  if (p.window > 0) return (p.window + p.group - 1) / p.group + 1;
  int64_t ns, ng, nr;
  state_of(p, p.max_tokens, &ns, &ng, &nr);
  return ng;
}

ko_layout layout_of(const ko_params& p) {
  const int64_t d = p.head_dim, G = p.group, b = p.bits;
  ko_layout L{};
  L.n_slots = slots_of(p);
  L.sink_k = 0;
  L.sink_v = L.sink_k + p.sinks * d * 4;
  L.res_k = L.sink_v + p.sinks * d * 4;
  L.res_v = L.res_k + p.residual * d * 2;
  L.groups = L.res_v + p.residual * d * 2;
  // group block: [K codes: G rows of d*b/8][K Δ row d, K min row d (fp16)]
  //              [V codes: d rows of G*b/8][V (Δ, min) per token (fp16)]
  L.blk_kq = 0;
  L.blk_ks = L.blk_kq + G * d * b / 8;
  L.blk_vq = L.blk_ks + 2 * d * 2;
  L.blk_vs = L.blk_vq + d * G * b / 8;
  // dense-and-sparse outliers (pigeon guide, "KVQuant adds": a small share
  // of the values, around one in a hundred, kept in fp16 beside the codes):
  // per block a key table and a value table in compressed sparse rows by
  // token: G + 1 u16 row pointers (entries of token t are [ptr[t], ptr[t+1])),
  // then n_outliers 4-byte entries from a 4-byte boundary, each table padded
  // to 16 bytes
  L.n_outliers = (static_cast<int64_t>(p.outlier_permille) * G * d + 999) / 1000;
  L.out_entries = L.n_outliers ? ((G + 1) * 2 + 3) / 4 * 4 : 0;
  const int64_t table = L.n_outliers ? (L.out_entries + 4 * L.n_outliers + 15) / 16 * 16 : 0;
  L.blk_ko = L.blk_vs + G * 2 * 2;
  L.blk_vo = L.blk_ko + table;
  L.block_bytes = L.blk_vo + table;
  L.unit_bytes = L.groups + L.n_slots * L.block_bytes;
  L.cache_bytes = static_cast<int64_t>(p.batch) * p.h_kv * L.unit_bytes;
  return L;
}

void put_f32(uint8_t* dst, float v) { std::memcpy(dst, &v, 4); }
float get_f32(const uint8_t* src) { float v; std::memcpy(&v, src, 4); return v; }
void put_u16(uint8_t* dst, uint16_t v) { dst[0] = static_cast<uint8_t>(v); dst[1] = static_cast<uint8_t>(v >> 8); }
uint16_t get_u16(const uint8_t* src) { return static_cast<uint16_t>(src[0] | (src[1] << 8)); }

}  // namespace

// ---------------------------------------------------------------------------
// The cache: a host byte arena laid out exactly like the device arena's cache
// region, plus the token count.  Tokens enter one at a time.
// ---------------------------------------------------------------------------
struct ko_cache {
  ko_params p;
  ko_layout L;
  std::vector<uint8_t> arena;
  int64_t T = 0;         // tokens appended so far (per sequence)
  int64_t n_groups = 0;  // frozen groups written so far
  int64_t n_res = 0;     // tokens live in the residual ring
};

namespace {

uint8_t* unit_ptr(ko_cache& c, int64_t b, int64_t h) {
  return c.arena.data() + (b * c.p.h_kv + h) * c.L.unit_bytes;
}
const uint8_t* unit_ptr(const ko_cache& c, int64_t b, int64_t h) {
  return c.arena.data() + (b * c.p.h_kv + h) * c.L.unit_bytes;
}

// The n largest |x| of x[0..len) (fp16; magnitude order is the order of the
// bit patterns without the sign), ties to the smaller index, flagged in skip.
void select_outliers(const uint16_t* x, int len, int64_t n, uint8_t* skip) {
  if (n <= 0) return;
  std::vector<int> idx(len);
  for (int i = 0; i < len; ++i) idx[i] = i;
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return (x[a] & 0x7FFF) > (x[b] & 0x7FFF); });
  for (int64_t k = 0; k < n && k < len; ++k) skip[idx[k]] = 1;
}

// The flagged values of a [G][d] block as a table of rows by token: row
// pointers ptr[0..G] (ptr[t] = entries of tokens before t), then at
// entries_off the {u8 t, u8 ch, fp16 x} entries in flat-index (t d + ch)
// order.
void write_table(const uint16_t* x, const uint8_t* skip, int G, int d, int64_t entries_off, uint8_t* out) {
  int64_t e = 0;
  for (int t = 0; t < G; ++t) {
    put_u16(out + 2 * t, static_cast<uint16_t>(e));
    for (int ch = 0; ch < d; ++ch) {
      if (!skip[t * d + ch]) continue;
      uint8_t* en = out + entries_off + 4 * e;
      en[0] = static_cast<uint8_t>(t);
      en[1] = static_cast<uint8_t>(ch);
      put_u16(en + 2, x[t * d + ch]);
      ++e;
    }
  }
  put_u16(out + 2 * G, static_cast<uint16_t>(e));
}

// Flush: the ring's oldest G tokens (absolute positions a0 .. a0+G-1) become
// frozen group g.  Keys: one (Δ, min) per channel over the G tokens; values:
// one (Δ, min) per token over the d channels.
void flush_group(ko_cache& c, uint8_t* unit, int64_t g) {
  const ko_params& p = c.p;
  const int d = p.head_dim, G = p.group, b = p.bits, R = p.residual, S = p.sinks;
  const int64_t a0 = S + g * G;
  const int64_t slot = g % c.L.n_slots;
  uint8_t* blk = unit + c.L.groups + slot * c.L.block_bytes;
  // gather the group's fp16 tokens from the ring: [G][d]
  std::vector<uint16_t> kx(static_cast<size_t>(G) * d), vx(static_cast<size_t>(G) * d);
  for (int t = 0; t < G; ++t) {
    const int64_t ring_slot = (a0 + t - S) % R;
    for (int ch = 0; ch < d; ++ch) {
      kx[t * d + ch] = get_u16(unit + c.L.res_k + (ring_slot * d + ch) * 2);
      vx[t * d + ch] = get_u16(unit + c.L.res_v + (ring_slot * d + ch) * 2);
    }
  }
  // outliers (dense-and-sparse): per block the n_outliers values of largest
  // magnitude, ties to the smaller flat index t d + ch, stored exactly in
  // index order and left out of the dense quantization
  const int64_t no = c.L.n_outliers;
  std::vector<uint8_t> kskip(static_cast<size_t>(G) * d, 0), vskip(static_cast<size_t>(G) * d, 0);
  select_outliers(kx.data(), G * d, no, kskip.data());
  select_outliers(vx.data(), G * d, no, vskip.data());
  if (no) {
    write_table(kx.data(), kskip.data(), G, d, c.L.out_entries, blk + c.L.blk_ko);
    write_table(vx.data(), vskip.data(), G, d, c.L.out_entries, blk + c.L.blk_vo);
  }
  // keys, per channel over the group's tokens
  std::vector<uint8_t> kcodes(static_cast<size_t>(G) * d);
  std::vector<uint8_t> col(G);
  for (int ch = 0; ch < d; ++ch) {
    uint16_t d16, mn16;
    quantize(&kx[ch], G, d, b, col.data(), &d16, &mn16, no ? &kskip[ch] : nullptr);
    for (int t = 0; t < G; ++t) kcodes[t * d + ch] = col[t];
    put_u16(blk + c.L.blk_ks + ch * 2, d16);
    put_u16(blk + c.L.blk_ks + (d + ch) * 2, mn16);
  }
  for (int t = 0; t < G; ++t)   // key rows are token-major: row t = d channels
    pack_row(&kcodes[t * d], d, b, blk + c.L.blk_kq + static_cast<int64_t>(t) * d * b / 8);
  // values, per token over the channels
  std::vector<uint8_t> vcodes(static_cast<size_t>(G) * d);
  for (int t = 0; t < G; ++t) {
    uint16_t d16, mn16;
    quantize(&vx[t * d], d, 1, b, &vcodes[t * d], &d16, &mn16, no ? &vskip[t * d] : nullptr);
    put_u16(blk + c.L.blk_vs + (t * 2 + 0) * 2, d16);
    put_u16(blk + c.L.blk_vs + (t * 2 + 1) * 2, mn16);
  }
  // value rows are channel-major inside the block: row ch = the group's G tokens
  std::vector<uint8_t> vrow(G);
  for (int ch = 0; ch < d; ++ch) {
    for (int t = 0; t < G; ++t) vrow[t] = vcodes[t * d + ch];
    pack_row(vrow.data(), G, b, blk + c.L.blk_vq + static_cast<int64_t>(ch) * G * b / 8);
  }
}

// Dequantized keys/values of every token of one unit, fp64, and which tokens
// the cache still holds (res[a] = 0 once a's group slot was overwritten).
void dequant_resident(const ko_cache& c, int64_t b_idx, int64_t h, double* K, double* V, uint8_t* res) {
  const ko_params& p = c.p;
  const int d = p.head_dim, G = p.group, b = p.bits, R = p.residual, S = p.sinks;
  const uint8_t* unit = unit_ptr(c, b_idx, h);
  const int64_t T = c.T;
  std::vector<uint8_t> row(std::max(d, G));
  for (int64_t a = 0; a < T; ++a) {
    double* kr = K + a * d;
    double* vr = V + a * d;
    res[a] = 0;
    if (a < S) {   // sink: fp32 as stored, always visible
      for (int ch = 0; ch < d; ++ch) {
        kr[ch] = get_f32(unit + c.L.sink_k + (a * d + ch) * 4);
        vr[ch] = get_f32(unit + c.L.sink_v + (a * d + ch) * 4);
      }
      res[a] = 1;
      continue;
    }
    const int64_t g = (a - S) / G;
    if (g < c.n_groups) {   // frozen group
      const int64_t slot = g % c.L.n_slots;
      const bool overwritten = (c.n_groups - 1 - g) >= c.L.n_slots;
      if (overwritten) { std::fill(kr, kr + d, 0.0); std::fill(vr, vr + d, 0.0); continue; }
      const uint8_t* blk = unit + c.L.groups + slot * c.L.block_bytes;
      const int t = static_cast<int>((a - S) - g * G);
      unpack_row(blk + c.L.blk_kq + static_cast<int64_t>(t) * d * b / 8, d, b, row.data());
      for (int ch = 0; ch < d; ++ch) {
        const double dq = f16_to_f32(get_u16(blk + c.L.blk_ks + ch * 2));
        const double mn = f16_to_f32(get_u16(blk + c.L.blk_ks + (d + ch) * 2));
        kr[ch] = mn + static_cast<double>(row[ch]) * dq;
      }
      const double vdq = f16_to_f32(get_u16(blk + c.L.blk_vs + (t * 2 + 0) * 2));
      const double vmn = f16_to_f32(get_u16(blk + c.L.blk_vs + (t * 2 + 1) * 2));
      for (int ch = 0; ch < d; ++ch) {
        unpack_row(blk + c.L.blk_vq + static_cast<int64_t>(ch) * G * b / 8, G, b, row.data());
        vr[ch] = vmn + static_cast<double>(row[t]) * vdq;
      }
      // outliers are exact (dense-and-sparse)
      for (int64_t e = 0; e < c.L.n_outliers; ++e) {
        const uint8_t* ke = blk + c.L.blk_ko + c.L.out_entries + 4 * e;
        if (ke[0] == t) kr[ke[1]] = f16_to_f32(get_u16(ke + 2));
        const uint8_t* ve = blk + c.L.blk_vo + c.L.out_entries + 4 * e;
        if (ve[0] == t) vr[ve[1]] = f16_to_f32(get_u16(ve + 2));
      }
    } else {   // residual ring, fp16
      const int64_t ring_slot = (a - S) % R;
      for (int ch = 0; ch < d; ++ch) {
        kr[ch] = f16_to_f32(get_u16(unit + c.L.res_k + (ring_slot * d + ch) * 2));
        vr[ch] = f16_to_f32(get_u16(unit + c.L.res_v + (ring_slot * d + ch) * 2));
      }
    }
    res[a] = 1;
  }
}

// Dequantized keys/values of one unit plus visibility for a query at the
// newest position T - 1.  Reading (window_mode 0): with a window, sinks stay
// visible and every other token is visible when it is among the most recent W
// tokens.  window_mode 1 (a pure window): the sinks too are visible only while
// they are among the most recent W tokens.
void dequant_unit(const ko_cache& c, int64_t b_idx, int64_t h, double* K, double* V, uint8_t* vis) {
  dequant_resident(c, b_idx, h, K, V, vis);
  const int64_t lo = (c.p.window > 0) ? c.T - c.p.window : 0;   // window start
  const int64_t from = c.p.window_mode == 1 ? 0 : c.p.sinks;     // tokens the window can expire
  for (int64_t a = from; a < c.T; ++a)
    if (a < lo) vis[a] = 0;
}

// Pre-RoPE keys (pigeon guide, "KVQuant adds": keys quantized before the
// rotary embedding, which would otherwise mix channel pairs): the rows K[a]
// of positions a = 0 .. T-1, as dequantized, rotated in place by RoPE at
// their own positions.  Reading: the rotate-half pairing, channel i with
// i + d/2, angle a * base^(-2i/d); the query arrives already rotated at its
// own position, so the scores are q . R(a) k_a.
void rope_rotate(const ko_params& p, double* K, int64_t T) {
  if (p.rope_base == 0.0) return;
  const int d = p.head_dim, h = d / 2;
  for (int i = 0; i < h; ++i) {
    const double theta = std::pow(p.rope_base, -2.0 * i / d);
    for (int64_t a = 0; a < T; ++a) {
      const double phi = static_cast<double>(a) * theta;
      const double cs = std::cos(phi), sn = std::sin(phi);
      const double x = K[a * d + i], y = K[a * d + i + h];
      K[a * d + i] = x * cs - y * sn;
      K[a * d + i + h] = y * cs + x * sn;
    }
  }
}

// softmax(q Kᵀ / sqrt(d)) V of one query row over the visible tokens, two
// passes in fp64 (scores and their max, then the weights); all zero when no
// token is visible.
void attend_row(const double* qd, const double* K, const double* V, const uint8_t* vis, int64_t T, int d,
                double* o) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(d));
  std::vector<double> s(static_cast<size_t>(T));
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t a = 0; a < T; ++a) {
    if (!vis[a]) continue;
    double acc = 0.0;
    for (int ch = 0; ch < d; ++ch) acc += qd[ch] * K[a * d + ch];
    s[a] = acc * inv_sqrt_d;
    m = std::max(m, s[a]);
  }
  double l = 0.0;
  std::vector<double> acc(d, 0.0);
  for (int64_t a = 0; a < T; ++a) {
    if (!vis[a]) continue;
    const double w = std::exp(s[a] - m);
    l += w;
    for (int ch = 0; ch < d; ++ch) acc[ch] += w * V[a * d + ch];
  }
  for (int ch = 0; ch < d; ++ch) o[ch] = (l > 0.0) ? acc[ch] / l : 0.0;
}

// fp64 decode attention of one unit (all query heads mapped to this kv head).
// Query head hq uses kv head floor(hq / (H_q / H_kv)) (contiguous GQA groups).
void attend_unit(const ko_cache& c, int64_t b_idx, int64_t h, const uint16_t* q, double* out) {
  const ko_params& p = c.p;
  const int d = p.head_dim;
  const int64_t T = c.T;
  const int rep = p.h_q / p.h_kv;
  std::vector<double> K(static_cast<size_t>(T) * d), V(static_cast<size_t>(T) * d);
  std::vector<uint8_t> vis(static_cast<size_t>(T));
  dequant_unit(c, b_idx, h, K.data(), V.data(), vis.data());
  rope_rotate(p, K.data(), T);
  std::vector<double> qd(d);
  for (int r = 0; r < rep; ++r) {
    const int64_t hq = h * rep + r;
    const uint16_t* qh = q + (b_idx * p.h_q + hq) * d;
    for (int ch = 0; ch < d; ++ch) qd[ch] = f16_to_f32(qh[ch]);
    attend_row(qd.data(), K.data(), V.data(), vis.data(), T, d, out + (b_idx * p.h_q + hq) * d);
  }
}

// fp64 causal attention of the M newest tokens of one unit as queries, over
// the cache as it stands (chunked prefill: the chunk was appended first, then
// each of its tokens attends to what precedes it and to itself; kvquant++
// README, long-document example, where prefill_chunk_size bounds each
// attention step while the context accumulates in the cache).
// Query j sits at position P = T - M + j; q and out are [B][M][H_q][d].
// Token a is visible to it when the cache still holds a, a <= P, and, with a
// window, a is a sink (window_mode 0 only) or among the W tokens ending at P.
// Tokens of the chunk
// are read as the cache holds them now (fp16 in the ring, codes once frozen).
void attend_unit_causal(const ko_cache& c, int64_t b_idx, int64_t h, const uint16_t* q, int64_t M,
                        double* out) {
  const ko_params& p = c.p;
  const int d = p.head_dim;
  const int64_t T = c.T, S = p.window_mode == 1 ? 0 : p.sinks;   // sinks that outlive the window
  const int rep = p.h_q / p.h_kv;
  std::vector<double> K(static_cast<size_t>(T) * d), V(static_cast<size_t>(T) * d);
  std::vector<uint8_t> res(static_cast<size_t>(T)), vis(static_cast<size_t>(T));
  dequant_resident(c, b_idx, h, K.data(), V.data(), res.data());
  rope_rotate(p, K.data(), T);
  std::vector<double> qd(d);
  for (int64_t j = 0; j < M; ++j) {
    const int64_t P = T - M + j;
    const int64_t lo = (p.window > 0) ? P + 1 - p.window : 0;
    for (int64_t a = 0; a < T; ++a) vis[a] = (res[a] && a <= P && (a < S || a >= lo)) ? 1 : 0;
    for (int r = 0; r < rep; ++r) {
      const int64_t row = (b_idx * M + j) * p.h_q + h * rep + r;
      for (int ch = 0; ch < d; ++ch) qd[ch] = f16_to_f32(q[row * d + ch]);
      attend_row(qd.data(), K.data(), V.data(), vis.data(), T, d, out + row * d);
    }
  }
}

}  // namespace

extern "C" {

uint16_t ko_f32_to_f16(float x) { return f32_to_f16(x); }
float ko_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
void ko_f32_to_f16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16(x[i]);
}
void ko_f16_to_f32_array(const uint16_t* h, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_to_f32(h[i]);
}

void ko_quantize(const uint16_t* x, int32_t n, int64_t stride, int32_t bits, uint8_t* codes,
                 uint16_t* delta16, uint16_t* min16) {
  quantize(x, n, stride, bits, codes, delta16, min16);
}

int ko_pack_row(const uint8_t* codes, int32_t L, int32_t bits, uint8_t* out) {
  if (bits < 1 || bits > 8) return kInvalid;
  return pack_row(codes, L, bits, out);
}
int ko_unpack_row(const uint8_t* packed, int32_t L, int32_t bits, uint8_t* codes) {
  if (bits < 1 || bits > 8) return kInvalid;
  return unpack_row(packed, L, bits, codes);
}

int ko_validate(const ko_params* p) { return p ? validate(*p) : kInvalid; }

int ko_layout_of(const ko_params* p, ko_layout* out) {
  if (!p || !out || validate(*p) != kOk) return kInvalid;
  *out = layout_of(*p);
  return kOk;
}

void ko_state_of(const ko_params* p, int64_t T, int64_t* n_sink, int64_t* n_groups, int64_t* n_res) {
  state_of(*p, T, n_sink, n_groups, n_res);
}

int ko_create(const ko_params* p, ko_cache** out) {
  if (!p || !out || validate(*p) != kOk) return kInvalid;
  ko_cache* c = new ko_cache();
  c->p = *p;
  c->L = layout_of(*p);
  c->arena.assign(static_cast<size_t>(c->L.cache_bytes), 0);
  *out = c;
  return kOk;
}

void ko_destroy(ko_cache* c) { delete c; }

// Tokens enter one at a time, in stream order, for every (batch, kv-head):
//   position a < S  -> fp32 sink slot a (keys and values);
//   otherwise       -> if the ring holds R tokens, its oldest G tokens are
//                      first flushed into frozen group n_groups; then the token
//                      is written to ring slot (a - S) mod R.
int ko_append(ko_cache* c, const uint16_t* k_new, const uint16_t* v_new, int64_t n) {
  if (!c || n < 0) return kInvalid;
  const ko_params& p = c->p;
  if (p.window == 0 && c->T + n > p.max_tokens) return kCapacity;
  const int d = p.head_dim, S = p.sinks, R = p.residual, G = p.group;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t a = c->T;
    const bool flush = (a >= S) && (c->n_res == R);
    for (int64_t b = 0; b < p.batch; ++b) {
      for (int64_t h = 0; h < p.h_kv; ++h) {
        uint8_t* unit = unit_ptr(*c, b, h);
        const uint16_t* kt = k_new + ((b * p.h_kv + h) * n + i) * d;
        const uint16_t* vt = v_new + ((b * p.h_kv + h) * n + i) * d;
        if (a < S) {
          for (int ch = 0; ch < d; ++ch) {
            put_f32(unit + c->L.sink_k + (a * d + ch) * 4, f16_to_f32(kt[ch]));
            put_f32(unit + c->L.sink_v + (a * d + ch) * 4, f16_to_f32(vt[ch]));
          }
          continue;
        }
        if (flush) flush_group(*c, unit, c->n_groups);
        const int64_t ring_slot = (a - S) % R;
        for (int ch = 0; ch < d; ++ch) {
          put_u16(unit + c->L.res_k + (ring_slot * d + ch) * 2, kt[ch]);
          put_u16(unit + c->L.res_v + (ring_slot * d + ch) * 2, vt[ch]);
        }
      }
    }
    if (a >= S) {
      if (flush) { c->n_groups += 1; c->n_res -= G; }
      c->n_res += 1;
    }
    c->T += 1;
  }
  return kOk;
}

int64_t ko_tokens(const ko_cache* c) { return c->T; }
int64_t ko_groups(const ko_cache* c) { return c->n_groups; }
int64_t ko_residual_count(const ko_cache* c) { return c->n_res; }
const uint8_t* ko_arena(const ko_cache* c) { return c->arena.data(); }

int ko_dequant_unit(const ko_cache* c, int32_t b, int32_t hkv, double* k_hat, double* v_hat,
                    uint8_t* visible) {
  if (!c || b < 0 || b >= c->p.batch || hkv < 0 || hkv >= c->p.h_kv) return kInvalid;
  dequant_unit(*c, b, hkv, k_hat, v_hat, visible);
  return kOk;
}

int ko_decode_attn(const ko_cache* c, const uint16_t* q, double* out, int32_t threads) {
  if (!c) return kInvalid;
  const int64_t units = static_cast<int64_t>(c->p.batch) * c->p.h_kv;
  const int nt = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(threads, units)));
  auto work = [&](int tid) {
    for (int64_t u = tid; u < units; u += nt) attend_unit(*c, u / c->p.h_kv, u % c->p.h_kv, q, out);
  };
  if (nt == 1) { work(0); return kOk; }
  std::vector<std::thread> pool;
  for (int t = 0; t < nt; ++t) pool.emplace_back(work, t);
  for (auto& th : pool) th.join();
  return kOk;
}

int ko_prefill_attn(const ko_cache* c, const uint16_t* q, int64_t n_queries, double* out, int32_t threads) {
  if (!c || n_queries < 1 || n_queries > c->T) return kInvalid;
  const int64_t units = static_cast<int64_t>(c->p.batch) * c->p.h_kv;
  const int nt = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(threads, units)));
  auto work = [&](int tid) {
    for (int64_t u = tid; u < units; u += nt)
      attend_unit_causal(*c, u / c->p.h_kv, u % c->p.h_kv, q, n_queries, out);
  };
  if (nt == 1) { work(0); return kOk; }
  std::vector<std::thread> pool;
  for (int t = 0; t < nt; ++t) pool.emplace_back(work, t);
  for (auto& th : pool) th.join();
  return kOk;
}

// Bytes a decode pass must move, per unit: packed codes of the visible
// quantized tokens (keys and values), the key (Δ, min) rows of every group
// touched, the value (Δ, min) of every visible quantized token, the fp16
// residual keys and values, the fp32 sinks, the key and value outlier tables
// (G + 1 u16 row pointers and n_outliers 4-byte entries each) of every group
// touched; plus q and out (fp16) per head.  Sinks count as visible (window_mode
// 0, the CUDA library's reading).
int64_t ko_decode_bytes(const ko_cache* c) {
  const ko_params& p = c->p;
  const int64_t d = p.head_dim, G = p.group, b = p.bits, S = p.sinks, T = c->T;
  const int64_t lo = (p.window > 0) ? std::max<int64_t>(T - p.window, 0) : 0;
  int64_t tq = 0, touched = 0;
  const int64_t first = std::max<int64_t>(0, c->n_groups - c->L.n_slots);
  for (int64_t g = first; g < c->n_groups; ++g) {
    const int64_t a0 = S + g * G, a1 = a0 + G;
    const int64_t vis = std::max<int64_t>(0, a1 - std::max(a0, lo));
    if (vis > 0) { tq += vis; touched += 1; }
  }
  const int64_t ns = std::min(T, S);
  const int64_t per_unit = 2 * tq * d * b / 8 + 4 * d * touched + 4 * tq + 4 * d * c->n_res + 8 * d * ns +
                          (c->L.n_outliers ? 2 * (2 * (G + 1) + 4 * c->L.n_outliers) * touched : 0);
  return per_unit * p.batch * p.h_kv + 4 * d * static_cast<int64_t>(p.batch) * p.h_q;
}

}  // extern "C"
