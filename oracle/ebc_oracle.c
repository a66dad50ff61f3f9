/*
 * ebc_oracle.c -- plain, slow, single-threaded CPU oracle of the
 * error-bounded embedding codec.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg are its only users.  The product path (the CUDA
 * library) never links or calls it, and the two share no source.
 *
 * Method source: "Accelerating Communication in Deep Learning Recommendation
 * Model Training with Dual-Level Adaptive Lossy Compression" (arXiv
 * 2407.04272v5), cited as [DLRM-EBLC].  The pages give the pipeline
 * (quantization encoder -> vector-based LZ -> Huffman, §III-D), the table-wise
 * and iteration-wise error bounds (§III-C, §IV-B) and the single-buffer
 * layout (§III-E, Fig. 7), but no formulas or formats; every step the pages
 * leave open is fixed here as a "reading" and written the same way in the
 * library's header comments.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fPIC -shared (no FMA
 * contraction, so every float operation below rounds once, as written).
 */
#include "ebc_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- format constants (the container specification, version 1) ---- */
#define O_RADIUS 128            /* bins q in (-R, R); sym = q + R          */
#define O_RADIUS_WIDE 512       /* the wide alphabet: 1024 symbols         */
#define O_MAX_SYMS 1024
#define O_LMAX 24               /* longest Huffman code                    */
#define O_MAGIC 0x31434245u     /* bytes 'E' 'B' 'C' '1'                   */
#define O_VERSION 2u
#define O_HEADER 144u
#define O_TABLE_REC 272u        /* eb, n_lit, n_match, n_out, 256 lengths  */
/* Bytes of a table record with an alphabet of A = 2R symbols: eb, counts, A lengths. */
static uint64_t table_rec(int R) { return 16u + 2u * (uint64_t)R; }
#define O_SEG_REC 16u           /* word_off, chunk_base, match_base, n_bits */
#define O_MAX_T 1024

static uint64_t pad16(uint64_t n) { return (n + 15u) & ~(uint64_t)15u; }
static int dim_ok(int D) { return D >= 4 && D <= 512 && (D & (D - 1)) == 0; }
/* Segment = run of consecutive batch rows of one table, padded to 128 bits in
 * the stream; about 8192 codes, and a whole number of 32-row bitmap words. */
static int64_t seg_rows(int D) { int64_t s = 8192 / D; return s < 32 ? 32 : s; }
/* Chunk = run of literal vectors of one segment decoded by one thread:
 * max(128, D) codes. */
static int64_t chunk_rows(int D) { int64_t k = 128 / D; return k < 1 ? 1 : k; }

static void wr16(uint8_t* p, uint32_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void wr32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static void wr64(uint8_t* p, uint64_t v) { wr32(p, (uint32_t)v); wr32(p + 4, (uint32_t)(v >> 32)); }
static uint32_t rd16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t rd32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static uint64_t rd64(const uint8_t* p) { return (uint64_t)rd32(p) | ((uint64_t)rd32(p + 4) << 32); }
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* An absolute bound is usable when eb and 2*eb are finite normal numbers and
 * the reciprocal 1/(2*eb) is a normal number too. */
static int eb_ok(float eb) {
  if (!(eb >= FLT_MIN) || !(eb <= FLT_MAX)) return 0;
  float ebx2 = 2.0f * eb;
  if (!(ebx2 <= FLT_MAX)) return 0;
  float inv = 1.0f / ebx2;
  return inv >= FLT_MIN;
}

/* ------------------------------------------------------------------------
 * Quantization encoder, [DLRM-EBLC] §III-D: each float becomes an integer bin
 * under the absolute bound eb.  The pages reject prediction for embedding
 * vectors (§III-B observation 1 and §III-D "Optimized Entropy Encoding", the
 * Lorenzo "false prediction" of Fig. 4), so the prediction is zero:
 *     q = round_half_even(x / (2 eb)),   xhat = q * 2 eb.
 * Reading: the division is a multiplication by the fp32 reciprocal of 2 eb,
 * and a bin is accepted only if |x - xhat| <= eb holds in fp32 and |q| < R;
 * otherwise the element is an outlier (sym 0) and its raw bits are kept.
 * ---------------------------------------------------------------------- */
static int quantize_one(float x, float eb, float ebx2, float inv, int R) {
  float t = x * inv;
  if (isnan(t) || fabsf(t) >= 1073741824.0f) return 0;
  float qf = nearbyintf(t);                 /* default mode: ties to even */
  int q = (int)qf;
  if (q <= -R || q >= R) return 0;
  float xhat = (float)q * ebx2;
  float err = fabsf(x - xhat);
  if (!(err <= eb)) return 0;
  return q + R;
}

int64_t ebo_quantize(const float* x, int64_t n, float eb, uint8_t* sym) {
  if (!eb_ok(eb) || n < 0) return -1;
  float ebx2 = 2.0f * eb, inv = 1.0f / ebx2;
  int64_t outl = 0;
  for (int64_t i = 0; i < n; ++i) {
    sym[i] = (uint8_t)quantize_one(x[i], eb, ebx2, inv, O_RADIUS);
    if (sym[i] == 0) ++outl;
  }
  return outl;
}

int64_t ebo_quantize_r(const float* x, int64_t n, float eb, int R, uint16_t* sym) {
  if (!eb_ok(eb) || n < 0 || (R != O_RADIUS && R != O_RADIUS_WIDE)) return -1;
  float ebx2 = 2.0f * eb, inv = 1.0f / ebx2;
  int64_t outl = 0;
  for (int64_t i = 0; i < n; ++i) {
    sym[i] = (uint16_t)quantize_one(x[i], eb, ebx2, inv, R);
    if (sym[i] == 0) ++outl;
  }
  return outl;
}

float ebo_dequantize(int sym, float eb) {
  float ebx2 = 2.0f * eb;
  return (float)(sym - O_RADIUS) * ebx2;
}

float ebo_dequantize_r(int sym, float eb, int R) {
  float ebx2 = 2.0f * eb;
  return (float)(sym - R) * ebx2;
}

/* ------------------------------------------------------------------------
 * Dedup key for the vector-based LZ encoder ([DLRM-EBLC] §III-D "Vector-based
 * LZ Encoding", §III-E "fixed pattern length"): the pattern is one whole
 * quantized embedding vector.  Reading: a 32-bit hash, the wrapping sum over
 * 4-code words w_k of lowbias32(w_k + k*0x9E3779B9) plus, for each outlier at
 * position d, lowbias32(raw_d ^ (d+1)*0x85EBCA6B).  A word packs its codes
 * little-endian: four 8-bit codes, or with the wide alphabet (16-bit codes)
 * two, so a vector has D/4 or D/2 words.  lowbias32 is C. Wellons'
 * published 32-bit integer mixer (xor-shift 16, multiply 0x7feb352d,
 * xor-shift 15, multiply 0x846ca68b, xor-shift 16).
 * ---------------------------------------------------------------------- */
static uint32_t lowbias32(uint32_t v) {
  v ^= v >> 16;
  v *= 0x7feb352dU;
  v ^= v >> 15;
  v *= 0x846ca68bU;
  v ^= v >> 16;
  return v;
}

uint32_t ebo_vector_hash(const uint8_t* sym, const float* x_row, int D) {
  uint32_t h = 0;
  for (int k = 0; k < D / 4; ++k) {
    uint32_t w = (uint32_t)sym[4 * k] | ((uint32_t)sym[4 * k + 1] << 8) |
                 ((uint32_t)sym[4 * k + 2] << 16) | ((uint32_t)sym[4 * k + 3] << 24);
    h += lowbias32(w + (uint32_t)k * 0x9E3779B9u);
  }
  for (int d = 0; d < D; ++d)
    if (sym[d] == 0) h += lowbias32(f2u(x_row[d]) ^ ((uint32_t)(d + 1) * 0x85EBCA6Bu));
  return h;
}

uint32_t ebo_vector_hash_r(const uint16_t* sym, const float* x_row, int D, int R) {
  uint32_t h = 0;
  if (R == O_RADIUS) {
    for (int k = 0; k < D / 4; ++k) {
      uint32_t w = (uint32_t)sym[4 * k] | ((uint32_t)sym[4 * k + 1] << 8) |
                   ((uint32_t)sym[4 * k + 2] << 16) | ((uint32_t)sym[4 * k + 3] << 24);
      h += lowbias32(w + (uint32_t)k * 0x9E3779B9u);
    }
  } else {
    for (int k = 0; k < D / 2; ++k) {
      uint32_t w = (uint32_t)sym[2 * k] | ((uint32_t)sym[2 * k + 1] << 16);
      h += lowbias32(w + (uint32_t)k * 0x9E3779B9u);
    }
  }
  for (int d = 0; d < D; ++d)
    if (sym[d] == 0) h += lowbias32(f2u(x_row[d]) ^ ((uint32_t)(d + 1) * 0x85EBCA6Bu));
  return h;
}

/* ------------------------------------------------------------------------
 * Huffman code lengths, [DLRM-EBLC] §III-D "Optimized Entropy Encoding"
 * (Huffman's minimum-redundancy code).  Reading, since the pages give no
 * tie rule: symbols with f > 0 sorted by (f, sym) ascending form the leaf
 * queue; merged nodes go to a FIFO queue; each pick takes the smaller front
 * and a tie goes to the leaf.  A single used symbol gets length 1.  If the
 * longest code exceeds lmax, every nonzero f becomes max(1, f >> 1) and the
 * code is rebuilt.
 * ---------------------------------------------------------------------- */
static int two_queue_lengths(const uint64_t* f, int A, uint8_t* len) {
  int order[O_MAX_SYMS], n = 0;
  memset(len, 0, (size_t)A);
  for (int s = 0; s < A; ++s)
    if (f[s] > 0) {
      /* insertion keeps (f, sym) order: equal f stay in sym order */
      int j = n++;
      while (j > 0 && f[order[j - 1]] > f[s]) { order[j] = order[j - 1]; --j; }
      order[j] = s;
    }
  if (n == 0) return 0;
  if (n == 1) { len[order[0]] = 1; return 1; }
  uint64_t node_w[O_MAX_SYMS - 1];
  int leaf_parent[O_MAX_SYMS], node_parent[O_MAX_SYMS - 1];
  int li = 0, qi = 0, qn = 0;
  for (int m = 0; m < n - 1; ++m) {
    uint64_t w = 0;
    for (int pick = 0; pick < 2; ++pick) {
      int leaf = li < n && (qi >= qn || f[order[li]] <= node_w[qi]);
      if (leaf) { leaf_parent[li] = m; w += f[order[li]]; ++li; }
      else { node_parent[qi] = m; w += node_w[qi]; ++qi; }
    }
    node_w[qn++] = w;
  }
  int depth[O_MAX_SYMS - 1];
  depth[n - 2] = 0;                       /* the last merge is the root */
  for (int m = n - 3; m >= 0; --m) depth[m] = depth[node_parent[m]] + 1;
  int maxlen = 0;
  for (int i = 0; i < n; ++i) {
    int l = depth[leaf_parent[i]] + 1;
    len[order[i]] = (uint8_t)(l > 255 ? 255 : l);
    if (l > maxlen) maxlen = l;
  }
  return maxlen;
}

int ebo_huffman_lengths_n(const uint64_t* freq, int A, int lmax, uint8_t* len) {
  if (lmax < 10 || lmax > 32 || A < 2 || A > O_MAX_SYMS) return -1;
  uint64_t f[O_MAX_SYMS];
  memcpy(f, freq, sizeof(uint64_t) * (size_t)A);
  for (int round = 0; round < 70; ++round) {
    if (two_queue_lengths(f, A, len) <= lmax) return round;
    for (int s = 0; s < A; ++s)
      if (f[s] > 0) f[s] = (f[s] >> 1) > 0 ? (f[s] >> 1) : 1;
  }
  return -1;
}

int ebo_huffman_lengths(const uint64_t* freq, int lmax, uint8_t* len) {
  if (lmax < 8 || lmax > 32) return -1;
  uint64_t f[256];
  memcpy(f, freq, sizeof f);
  for (int round = 0; round < 70; ++round) {
    if (two_queue_lengths(f, 256, len) <= lmax) return round;
    for (int s = 0; s < 256; ++s)
      if (f[s] > 0) f[s] = (f[s] >> 1) > 0 ? (f[s] >> 1) : 1;
  }
  return -1;
}

/* Canonical codes: lengths ascending, then symbols ascending, consecutive
 * values, the first code of each length being (previous first + count) << 1
 * (the DEFLATE rule). */
int ebo_canonical_codes_n(const uint8_t* len, int A, int lmax, uint32_t* code) {
  uint64_t count[33] = {0};
  if (lmax < 1 || lmax > 32 || A < 1 || A > O_MAX_SYMS) return -1;
  for (int s = 0; s < A; ++s) {
    if (len[s] > lmax) return -1;
    count[len[s]]++;
  }
  count[0] = 0;
  uint64_t kraft = 0;
  for (int l = 1; l <= lmax; ++l) kraft += count[l] << (lmax - l);
  if (kraft > ((uint64_t)1 << lmax)) return -1;
  uint64_t next[33];
  uint64_t c = 0;
  next[0] = 0;
  for (int l = 1; l <= lmax; ++l) { c = (c + count[l - 1]) << 1; next[l] = c; }
  for (int s = 0; s < A; ++s) code[s] = len[s] ? (uint32_t)next[len[s]]++ : 0u;
  return 0;
}

int ebo_canonical_codes(const uint8_t* len, int lmax, uint32_t* code) {
  return ebo_canonical_codes_n(len, 256, lmax, code);
}

/* ------------------------------------------------------------------------
 * Iteration-wise error-bound decay, [DLRM-EBLC] §III-C "Iteration-wise
 * Configuration" (decay phase then constant phase; logarithmic or stepwise
 * decay, stepwise the default) and §IV-B Fig. 10 ("Decay_2x": 2x base down to
 * base; "Drop_2x": 2x base until the end of the initial phase, then base).
 * Reading: the factor multiplies the base bound and does not compound;
 * m0 is the initial multiplier, phase_len P the decay phase, n_steps S the
 * stairs of the stepwise form:
 *   linear     m0 - (m0-1) * (i/P)                    (i < P)
 *   stepwise   m0 - (m0-1) * floor(i*S/P) / S          (i < P)
 *   drop       m0                                       (i < P)
 *   log        m0^(1 - i/P)                             (i < P)
 * and 1 for i >= P, for "none", or when P <= 0.
 * ---------------------------------------------------------------------- */
double ebo_decay_factor(int fn, int64_t iter, double m0, int64_t P, int S) {
  if (fn == 0 || P <= 0 || iter >= P) return 1.0;
  if (iter < 0) iter = 0;
  double frac = (double)iter / (double)P;
  switch (fn) {
    case 1: return m0 - (m0 - 1.0) * frac;
    case 2: {
      if (S < 1) S = 1;
      int64_t k = (iter * (int64_t)S) / P;
      return m0 - (m0 - 1.0) * ((double)k / (double)S);
    }
    case 3: return m0;
    case 4: return pow(m0, 1.0 - frac);
    default: return 1.0;
  }
}

/* ------------------------------------------------------------------------
 * Container layout (all little-endian, sections 16-byte aligned):
 *   header (144 B) | T table records (272 B) | T*nseg segment records (16 B)
 *   | match bitmap T*ceil(B/32) u32 | chunk lengths u16 | refs u16/u32
 *   | bitstream u32 words
 * An outlier is coded inline: the code of symbol 0, then the 32 raw bits of
 * the value, MSB first.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint64_t off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;
} layout_t;

static layout_t make_layout(int64_t B, int T, int D, uint64_t n_chunks, uint64_t n_match,
                            uint64_t words, int ref_bytes, uint64_t rec_bytes) {
  layout_t L;
  int64_t nseg = (B + seg_rows(D) - 1) / seg_rows(D);
  int64_t nw = (B + 31) / 32;
  L.off_seg = O_HEADER + (uint64_t)T * rec_bytes;
  L.off_bitmap = L.off_seg + (uint64_t)T * (uint64_t)nseg * O_SEG_REC;
  L.off_chunks = L.off_bitmap + pad16((uint64_t)T * (uint64_t)nw * 4u);
  L.off_refs = L.off_chunks + pad16(n_chunks * 2u);
  L.off_bits = L.off_refs + pad16(n_match * (uint64_t)ref_bytes);
  L.total = L.off_bits + words * 4u;
  return L;
}

static int shape_ok(int64_t B, int T, int D) {
  if (B < 0 || T < 0 || T > O_MAX_T || !dim_ok(D)) return 0;
  if (B > 16777215) return 0;
  if ((uint64_t)B * (uint64_t)T * (uint64_t)D > ((uint64_t)1 << 31)) return 0;
  return 1;
}

uint64_t ebo_compress_bound_r(int64_t B, int T, int D, int R) {
  if (!shape_ok(B, T, D) || (R != O_RADIUS && R != O_RADIUS_WIDE)) return 0;
  uint64_t N = (uint64_t)B * T * D;
  int64_t nseg = (B + seg_rows(D) - 1) / seg_rows(D);
  uint64_t vec = (uint64_t)B * T;
  uint64_t words = (N * (O_LMAX + 32) + 31) / 32 + 4u * (uint64_t)T * (uint64_t)nseg;
  layout_t L = make_layout(B, T, D, vec, vec, words, B <= 65536 ? 2 : 4, table_rec(R));
  return L.total;
}

uint64_t ebo_compress_bound(int64_t B, int T, int D) { return ebo_compress_bound_r(B, T, D, O_RADIUS); }

/* MSB-first bit writer over u32 words: bit i lives in word i/32 at bit 31-i%32. */
static void put_bits(uint32_t* words, uint64_t* pos, uint32_t code, int len) {
  for (int i = len - 1; i >= 0; --i) {
    uint32_t bit = (code >> i) & 1u;
    words[*pos >> 5] |= bit << (31 - (*pos & 31));
    ++*pos;
  }
}

typedef struct { uint32_t h; uint32_t b; } hb_t;
static int cmp_hb(const void* a, const void* c) {
  const hb_t* x = (const hb_t*)a; const hb_t* y = (const hb_t*)c;
  if (x->h != y->h) return x->h < y->h ? -1 : 1;
  return x->b < y->b ? -1 : (x->b > y->b);
}

int ebo_compress(const float* x, int64_t B, int T, int D, const float* eb, uint8_t* out,
                 uint64_t cap, ebo_info* info, uint8_t* sym_out, uint32_t* ref_out,
                 uint8_t* lens_out) {
  return ebo_compress_modes(x, B, T, D, eb, NULL, out, cap, info, sym_out, ref_out, lens_out);
}

int ebo_compress_modes(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes,
                       uint8_t* out, uint64_t cap, ebo_info* info, uint8_t* sym_out, uint32_t* ref_out,
                       uint8_t* lens_out) {
  return ebo_compress_ex(x, B, T, D, eb, modes, 0, out, cap, info, sym_out, ref_out, lens_out);
}

static int compress_impl(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes,
                         int window, int R, uint8_t* out, uint64_t cap, ebo_info* info, uint16_t* sym_out,
                         uint32_t* ref_out, uint8_t* lens_out);

int ebo_compress_ex(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes, int window,
                    uint8_t* out, uint64_t cap, ebo_info* info, uint8_t* sym_out, uint32_t* ref_out,
                    uint8_t* lens_out) {
  if (!shape_ok(B, T, D)) return EBO_ERR_INVALID_ARG;
  const size_t N = (size_t)B * (size_t)T * (size_t)D;
  uint16_t* s16 = sym_out ? (uint16_t*)malloc((N ? N : 1) * 2) : NULL;
  if (sym_out && !s16) return EBO_ERR_INVALID_ARG;
  const int rc = compress_impl(x, B, T, D, eb, modes, window, O_RADIUS, out, cap, info, s16, ref_out, lens_out);
  if (s16) {
    if (rc == EBO_OK || rc == EBO_ERR_CAPACITY)
      for (size_t i = 0; i < N; ++i) sym_out[i] = (uint8_t)s16[i];
    free(s16);
  }
  return rc;
}

int ebo_compress_r(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes, int window,
                   int R, uint8_t* out, uint64_t cap, ebo_info* info, uint16_t* sym_out, uint32_t* ref_out,
                   uint8_t* lens_out) {
  return compress_impl(x, B, T, D, eb, modes, window, R, out, cap, info, sym_out, ref_out, lens_out);
}

/* The whole encoder with radius R: 128 (8-bit codes, the default) or 512 (the
 * wide alphabet, 1024 symbols, 16-bit codes).  lens_out is [T][2R]. */
static int compress_impl(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes,
                         int window, int R, uint8_t* out, uint64_t cap, ebo_info* info, uint16_t* sym_out,
                         uint32_t* ref_out, uint8_t* lens_out) {
  if (!shape_ok(B, T, D) || window < 0 || window > EBO_MAX_WINDOW || (R != O_RADIUS && R != O_RADIUS_WIDE))
    return EBO_ERR_INVALID_ARG;
  const int A = 2 * R;                                      /* symbols: 0 (outlier) and q + R */
  const uint64_t REC = table_rec(R);
  for (int t = 0; t < T; ++t)
    if (!eb_ok(eb[t]) || (modes && modes[t] > 3)) return EBO_ERR_INVALID_ARG;
  const int64_t SB = seg_rows(D), KC = chunk_rows(D);
  const int64_t nseg = (B + SB - 1) / SB, nw = (B + 31) / 32;
  const int ref_bytes = window > 0 ? 1 : (B <= 65536 ? 2 : 4);
  const size_t nvec = (size_t)B * (size_t)T;
  const size_t N = nvec * (size_t)D;

  uint16_t* sym = (uint16_t*)malloc((N ? N : 1) * 2);    /* [T][B][D] */
  uint32_t* hash = (uint32_t*)malloc((nvec ? nvec : 1) * 4);
  uint32_t* ref = (uint32_t*)malloc((nvec ? nvec : 1) * 4);
  uint8_t* lens = (uint8_t*)calloc((size_t)(T ? T : 1) * (size_t)A, 1);
  uint32_t* codes = (uint32_t*)calloc((size_t)(T ? T : 1) * (size_t)A, 4);
  hb_t* pairs = (hb_t*)malloc((size_t)(B ? B : 1) * sizeof(hb_t));
  if (!sym || !hash || !ref || !lens || !codes || !pairs) {
    free(sym); free(hash); free(ref); free(lens); free(codes); free(pairs);
    return EBO_ERR_INVALID_ARG;
  }

  /* 1. quantization codes, table-major */
  for (int t = 0; t < T; ++t) {
    float ebx2 = 2.0f * eb[t], inv = 1.0f / ebx2;
    for (int64_t b = 0; b < B; ++b)
      for (int d = 0; d < D; ++d)
        sym[((size_t)t * B + b) * D + d] =
            (uint16_t)quantize_one(x[((size_t)b * T + t) * D + d], eb[t], ebx2, inv, R);
  }
  /* 2. vector hashes */
  for (int t = 0; t < T; ++t)
    for (int64_t b = 0; b < B; ++b)
      hash[(size_t)t * B + b] =
          ebo_vector_hash_r(sym + ((size_t)t * B + b) * D, x + ((size_t)b * T + t) * D, D, R);
  /* 3. vector dedup ([DLRM-EBLC] §III-D / §III-E, vector-based LZ).  Reading:
   * the window is the whole batch of one table and the reference is the first
   * occurrence, ref(b) = min{b' : hash(b') = hash(b)}; b is a match when
   * ref(b) < b and both vectors have the same codes and the same raw bits at
   * outliers, else a literal.  References therefore always name literals. */
  for (int t = 0; t < T; ++t) {
    if (modes && (modes[t] & EBO_MODE_NO_DEDUP)) {   /* the table's vectors are all literals */
      for (int64_t b = 0; b < B; ++b) ref[(size_t)t * B + b] = (uint32_t)b;
      continue;
    }
    if (window > 0) {
      /* sliding window ([DLRM-EBLC] §III-E "extended window size", §IV-D Table VI): the
       * reference is the nearest earlier row within `window` rows with the same hash; b is a
       * match when it also has the same codes and raw outlier bits, else a literal.  A
       * reference may itself be a match (chains end at a literal). */
      for (int64_t b = 0; b < B; ++b) {
        const uint32_t hb = hash[(size_t)t * B + b];
        int64_t r = b;
        for (int64_t c2 = b - 1; c2 >= 0 && c2 >= b - window; --c2)
          if (hash[(size_t)t * B + c2] == hb) { r = c2; break; }
        int match = 0;
        if (r < b) {
          const uint16_t* sb = sym + ((size_t)t * B + b) * D;
          const uint16_t* sr = sym + ((size_t)t * B + r) * D;
          const float* xb = x + ((size_t)b * T + t) * D;
          const float* xr = x + ((size_t)r * T + t) * D;
          match = memcmp(sb, sr, (size_t)D * 2) == 0;
          for (int d = 0; match && d < D; ++d)
            if (sb[d] == 0 && f2u(xb[d]) != f2u(xr[d])) match = 0;
        }
        ref[(size_t)t * B + b] = match ? (uint32_t)r : (uint32_t)b;
      }
      continue;
    }
    for (int64_t b = 0; b < B; ++b) { pairs[b].h = hash[(size_t)t * B + b]; pairs[b].b = (uint32_t)b; }
    qsort(pairs, (size_t)B, sizeof(hb_t), cmp_hb);
    for (int64_t i = 0; i < B; ++i) {
      int64_t g = i;
      while (g > 0 && pairs[g - 1].h == pairs[i].h) --g;
      uint32_t b = pairs[i].b, r = pairs[g].b;
      int match = 0;
      if (r < b) {
        const uint16_t* sb = sym + ((size_t)t * B + b) * D;
        const uint16_t* sr = sym + ((size_t)t * B + r) * D;
        const float* xb = x + ((size_t)b * T + t) * D;
        const float* xr = x + ((size_t)r * T + t) * D;
        match = memcmp(sb, sr, (size_t)D * 2) == 0;
        for (int d = 0; match && d < D; ++d)
          if (sb[d] == 0 && f2u(xb[d]) != f2u(xr[d])) match = 0;
      }
      ref[(size_t)t * B + b] = match ? r : b;
    }
  }
  /* 4. per-table histogram of literal codes, Huffman lengths, canonical codes */
  for (int t = 0; t < T; ++t) {
    uint64_t f[O_MAX_SYMS] = {0};
    for (int64_t b = 0; b < B; ++b)
      if (ref[(size_t)t * B + b] == (uint32_t)b)
        for (int d = 0; d < D; ++d) f[sym[((size_t)t * B + b) * D + d]]++;
    if (modes && (modes[t] & EBO_MODE_RAW_CODES)) {
      /* raw codes: every symbol log2(A) bits, 8 or 10 (the canonical code of symbol s is s) */
      memset(lens + (size_t)t * A, A == 256 ? 8 : 10, (size_t)A);
    } else if (ebo_huffman_lengths_n(f, A, O_LMAX, lens + (size_t)t * A) < 0) {
      free(sym); free(hash); free(ref); free(lens); free(codes); free(pairs);
      return EBO_ERR_INVALID_ARG;
    }
    if (ebo_canonical_codes_n(lens + (size_t)t * A, A, O_LMAX, codes + (size_t)t * A) < 0) {
      free(sym); free(hash); free(ref); free(lens); free(codes); free(pairs);
      return EBO_ERR_INVALID_ARG;
    }
  }
  /* 5. sizes */
  uint64_t n_lit = 0, n_match = 0, n_out = 0, n_chunks = 0, words = 0;
  for (int t = 0; t < T; ++t)
    for (int64_t s = 0; s < nseg; ++s) {
      uint64_t lits = 0, bits = 0;
      for (int64_t b = s * SB; b < B && b < (s + 1) * SB; ++b) {
        if (ref[(size_t)t * B + b] != (uint32_t)b) { ++n_match; continue; }
        ++lits;
        for (int d = 0; d < D; ++d) {
          uint16_t c = sym[((size_t)t * B + b) * D + d];
          bits += lens[(size_t)t * A + c];
          if (c == 0) { ++n_out; bits += 32; }
        }
      }
      n_lit += lits;
      n_chunks += (lits + (uint64_t)KC - 1) / (uint64_t)KC;
      words += ((bits + 127) / 128) * 4;
    }
  layout_t L = make_layout(B, T, D, n_chunks, n_match, words, ref_bytes, REC);
  if (info) {
    info->n_literal = n_lit; info->n_match = n_match; info->n_outlier = n_out;
    info->n_chunks = n_chunks; info->bitstream_bytes = words * 4; info->total_bytes = L.total;
  }
  if (sym_out) memcpy(sym_out, sym, N * 2);
  if (ref_out) memcpy(ref_out, ref, nvec * 4);
  if (lens_out) memcpy(lens_out, lens, (size_t)T * (size_t)A);
  if (L.total > cap) {
    free(sym); free(hash); free(ref); free(lens); free(codes); free(pairs);
    return EBO_ERR_CAPACITY;
  }

  /* 6. write the container */
  memset(out, 0, (size_t)L.total);
  uint8_t* h = out;
  wr32(h + 0, O_MAGIC); wr32(h + 4, O_VERSION); wr64(h + 8, (uint64_t)B);
  wr32(h + 16, (uint32_t)T); wr32(h + 20, (uint32_t)D); wr32(h + 24, (uint32_t)R);
  wr32(h + 28, O_LMAX); wr32(h + 32, (uint32_t)SB); wr32(h + 36, (uint32_t)KC);
  wr32(h + 40, (uint32_t)ref_bytes); wr32(h + 44, (uint32_t)window);
  wr64(h + 48, n_lit); wr64(h + 56, n_match); wr64(h + 64, n_out); wr64(h + 72, n_chunks);
  wr64(h + 80, words); wr64(h + 88, L.off_seg); wr64(h + 96, L.off_bitmap);
  wr64(h + 104, L.off_chunks); wr64(h + 112, L.off_refs); wr64(h + 120, L.off_bits);
  wr64(h + 128, L.total); wr64(h + 136, 0);

  uint32_t* stream = (uint32_t*)calloc((size_t)(words ? words : 1), 4);
  uint64_t chunk_i = 0, match_i = 0, word_i = 0;
  for (int t = 0; t < T; ++t) {
    uint8_t* rec = out + O_HEADER + (size_t)t * REC;
    uint32_t tl = 0, tm = 0, to = 0;
    for (int64_t s = 0; s < nseg; ++s) {
      uint8_t* srec = out + L.off_seg + ((size_t)t * nseg + s) * O_SEG_REC;
      wr32(srec + 0, (uint32_t)word_i); wr32(srec + 4, (uint32_t)chunk_i);
      wr32(srec + 8, (uint32_t)match_i);
      uint64_t pos = word_i * 32, lit_in_seg = 0, chunk_start = pos;
      int64_t b_end = (s + 1) * SB < B ? (s + 1) * SB : B;
      for (int64_t b = s * SB; b < b_end; ++b) {
        uint32_t r = ref[(size_t)t * B + b];
        if (r != (uint32_t)b) {
          uint8_t* bm = out + L.off_bitmap + ((size_t)t * nw + (size_t)(b >> 5)) * 4;
          wr32(bm, rd32(bm) | (1u << (b & 31)));
          if (window > 0) out[L.off_refs + match_i] = (uint8_t)((uint32_t)b - r);   /* distance */
          else if (ref_bytes == 2) wr16(out + L.off_refs + match_i * 2, r);
          else wr32(out + L.off_refs + match_i * 4, r);
          ++match_i; ++tm;
          continue;
        }
        const uint16_t* sv = sym + ((size_t)t * B + b) * D;
        const float* xv = x + ((size_t)b * T + t) * D;
        for (int d = 0; d < D; ++d) {
          put_bits(stream, &pos, codes[(size_t)t * A + sv[d]], lens[(size_t)t * A + sv[d]]);
          if (sv[d] == 0) { put_bits(stream, &pos, f2u(xv[d]), 32); ++to; }
        }
        ++lit_in_seg; ++tl;
        if (lit_in_seg % (uint64_t)KC == 0) {        /* a chunk holds KC literals */
          wr16(out + L.off_chunks + chunk_i * 2, (uint32_t)(pos - chunk_start));
          ++chunk_i; chunk_start = pos;
        }
      }
      if (lit_in_seg % (uint64_t)KC != 0) {          /* the segment's last, short chunk */
        wr16(out + L.off_chunks + chunk_i * 2, (uint32_t)(pos - chunk_start));
        ++chunk_i; chunk_start = pos;
      }
      wr32(srec + 12, (uint32_t)(pos - word_i * 32));
      word_i += ((pos - word_i * 32 + 127) / 128) * 4;
    }
    wr32(rec + 0, f2u(eb[t])); wr32(rec + 4, tl); wr32(rec + 8, tm); wr32(rec + 12, to);
    memcpy(rec + 16, lens + (size_t)t * A, (size_t)A);
  }
  for (uint64_t w = 0; w < words; ++w) wr32(out + L.off_bits + w * 4, stream[w]);
  free(stream);
  free(sym); free(hash); free(ref); free(lens); free(codes); free(pairs);
  return EBO_OK;
}

/* ------------------------------------------------------------------------
 * Decoder: inverts the container; every read is bounds-checked and every
 * inconsistency is EBO_ERR_CORRUPT.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint32_t first[O_LMAX + 2];   /* first canonical code of each length  */
  uint32_t count[O_LMAX + 2];
  uint32_t offset[O_LMAX + 2];  /* index of that first code in sorted[] */
  uint16_t sorted[O_MAX_SYMS];  /* symbols by (length, symbol)          */
} dec_t;

static int build_decoder(const uint8_t* len, int A, dec_t* dc) {
  uint32_t code[O_MAX_SYMS];
  if (ebo_canonical_codes_n(len, A, O_LMAX, code) < 0) return -1;
  memset(dc, 0, sizeof *dc);
  for (int s = 0; s < A; ++s) dc->count[len[s]]++;
  dc->count[0] = 0;
  uint32_t k = 0;
  for (int l = 1; l <= O_LMAX; ++l) {
    dc->offset[l] = k;
    for (int s = 0; s < A; ++s)
      if (len[s] == l) {
        if (k == dc->offset[l]) dc->first[l] = code[s];
        dc->sorted[k++] = (uint16_t)s;
      }
  }
  return 0;
}

static int decompress_impl(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D, float* xhat,
                           uint16_t* sym_out, int* radius_out);

int ebo_decompress(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D, float* xhat,
                   uint8_t* sym_out) {
  if (!shape_ok(B, T, D)) return EBO_ERR_INVALID_ARG;
  const size_t N = (size_t)B * (size_t)T * (size_t)D;
  uint16_t* s16 = sym_out ? (uint16_t*)malloc((N ? N : 1) * 2) : NULL;
  if (sym_out && !s16) return EBO_ERR_INVALID_ARG;
  int R = 0;
  int rc = decompress_impl(in, in_bytes, B, T, D, xhat, s16, &R);
  if (s16) {
    if (rc == EBO_OK && R != O_RADIUS) rc = EBO_ERR_INVALID_ARG;   /* 16-bit codes: use ebo_decompress_r */
    if (rc == EBO_OK)
      for (size_t i = 0; i < N; ++i) sym_out[i] = (uint8_t)s16[i];
    free(s16);
  }
  return rc;
}

int ebo_decompress_r(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D, float* xhat,
                     uint16_t* sym_out) {
  int R = 0;
  return decompress_impl(in, in_bytes, B, T, D, xhat, sym_out, &R);
}

/* Decoder of containers with either radius (read from the header). */
static int decompress_impl(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D, float* xhat,
                           uint16_t* sym_out, int* radius_out) {
  if (!shape_ok(B, T, D)) return EBO_ERR_INVALID_ARG;
  if (in_bytes < O_HEADER) return EBO_ERR_CORRUPT;
  if (rd32(in) != O_MAGIC || rd32(in + 4) != O_VERSION) return EBO_ERR_CORRUPT;
  if (rd64(in + 8) != (uint64_t)B || rd32(in + 16) != (uint32_t)T || rd32(in + 20) != (uint32_t)D)
    return EBO_ERR_INVALID_ARG;
  const int64_t SB = seg_rows(D), KC = chunk_rows(D);
  const int64_t nseg = (B + SB - 1) / SB, nw = (B + 31) / 32;
  const uint32_t window = rd32(in + 44);   /* 0: whole-batch references; else distances */
  const int ref_bytes = window > 0 ? 1 : (B <= 65536 ? 2 : 4);
  const int R = (int)rd32(in + 24);
  if (R != O_RADIUS && R != O_RADIUS_WIDE) return EBO_ERR_CORRUPT;
  const int A = 2 * R;
  const uint64_t REC = table_rec(R);
  *radius_out = R;
  if (rd32(in + 28) != O_LMAX || rd32(in + 32) != (uint32_t)SB ||
      rd32(in + 36) != (uint32_t)KC || rd32(in + 40) != (uint32_t)ref_bytes || window > EBO_MAX_WINDOW)
    return EBO_ERR_CORRUPT;
  uint64_t n_lit = rd64(in + 48), n_match = rd64(in + 56), n_out = rd64(in + 64);
  uint64_t n_chunks = rd64(in + 72), words = rd64(in + 80);
  uint64_t nvec = (uint64_t)B * (uint64_t)T;
  if (n_lit + n_match != nvec || n_chunks > nvec || n_out > nvec * (uint64_t)D ||
      words > ((uint64_t)1 << 34))
    return EBO_ERR_CORRUPT;
  layout_t L = make_layout(B, T, D, n_chunks, n_match, words, ref_bytes, REC);
  if (rd64(in + 88) != L.off_seg || rd64(in + 96) != L.off_bitmap || rd64(in + 104) != L.off_chunks ||
      rd64(in + 112) != L.off_refs || rd64(in + 120) != L.off_bits || rd64(in + 128) != L.total ||
      rd64(in + 136) != 0 || L.total > in_bytes)
    return EBO_ERR_CORRUPT;

  const size_t N = (size_t)nvec * (size_t)D;
  uint16_t* sym = (uint16_t*)malloc((N ? N : 1) * 2);
  if (!sym) return EBO_ERR_INVALID_ARG;
  uint64_t chunk_i = 0, match_i = 0, out_i = 0, word_i = 0, lit_total = 0;
  int err = EBO_OK;
  for (int t = 0; t < T && err == EBO_OK; ++t) {
    const uint8_t* rec = in + O_HEADER + (size_t)t * REC;
    float eb = u2f(rd32(rec));
    if (!eb_ok(eb)) { err = EBO_ERR_CORRUPT; break; }
    dec_t dc;
    if (build_decoder(rec + 16, A, &dc) < 0) { err = EBO_ERR_CORRUPT; break; }
    uint32_t tl = 0, tm = 0, to = 0;
    for (int64_t s = 0; s < nseg && err == EBO_OK; ++s) {
      const uint8_t* srec = in + L.off_seg + ((size_t)t * nseg + s) * O_SEG_REC;
      if (rd32(srec) != word_i || rd32(srec + 4) != chunk_i || rd32(srec + 8) != match_i) {
        err = EBO_ERR_CORRUPT;
        break;
      }
      int64_t b_end = (s + 1) * SB < B ? (s + 1) * SB : B;
      uint64_t seg_bit0 = word_i * 32, pos = seg_bit0, lit_in_seg = 0, chunk_start = pos;
      uint64_t seg_lits = 0;
      for (int64_t b = s * SB; b < b_end; ++b) {
        const uint8_t* bm = in + L.off_bitmap + ((size_t)t * nw + (size_t)(b >> 5)) * 4;
        if (!((rd32(bm) >> (b & 31)) & 1u)) ++seg_lits;
      }
      for (int64_t b = s * SB; b < b_end && err == EBO_OK; ++b) {
        const uint8_t* bm = in + L.off_bitmap + ((size_t)t * nw + (size_t)(b >> 5)) * 4;
        if ((rd32(bm) >> (b & 31)) & 1u) { ++match_i; ++tm; continue; }
        if (chunk_i >= n_chunks) { err = EBO_ERR_CORRUPT; break; }
        uint64_t chunk_end = chunk_start + rd16(in + L.off_chunks + chunk_i * 2);
        uint16_t* sv = sym + ((size_t)t * B + b) * D;
        for (int d = 0; d < D; ++d) {
          uint32_t code = 0;
          int l = 0, found = 0;
          while (!found) {
            if (l >= O_LMAX || pos >= chunk_end || pos >= words * 32) { err = EBO_ERR_CORRUPT; break; }
            uint32_t word = rd32(in + L.off_bits + (pos >> 5) * 4);
            code = (code << 1) | ((word >> (31 - (pos & 31))) & 1u);
            ++pos; ++l;
            if (dc.count[l] && code >= dc.first[l] && code - dc.first[l] < dc.count[l]) {
              sv[d] = dc.sorted[dc.offset[l] + (code - dc.first[l])];
              found = 1;
            }
          }
          if (err) break;
          float v;
          if (sv[d] == 0) {
            uint32_t raw = 0;
            for (int k = 0; k < 32; ++k) {
              if (pos >= chunk_end || pos >= words * 32) { err = EBO_ERR_CORRUPT; break; }
              uint32_t word = rd32(in + L.off_bits + (pos >> 5) * 4);
              raw = (raw << 1) | ((word >> (31 - (pos & 31))) & 1u);
              ++pos;
            }
            if (err) break;
            v = u2f(raw);
            ++out_i; ++to;
          } else {
            v = ebo_dequantize_r(sv[d], eb, R);
          }
          xhat[((size_t)b * T + t) * D + d] = v;
        }
        if (err) break;
        ++lit_in_seg; ++tl; ++lit_total;
        if (lit_in_seg % (uint64_t)KC == 0 || lit_in_seg == seg_lits) {
          if (pos != chunk_end) { err = EBO_ERR_CORRUPT; break; }
          ++chunk_i; chunk_start = pos;
        }
      }
      if (err) break;
      /* bitmap bits past B must be clear */
      if (s == nseg - 1 && (B & 31)) {
        const uint8_t* bm = in + L.off_bitmap + ((size_t)t * nw + (size_t)(nw - 1)) * 4;
        if (rd32(bm) >> (B & 31)) { err = EBO_ERR_CORRUPT; break; }
      }
      if (rd32(srec + 12) != (uint32_t)(pos - seg_bit0)) { err = EBO_ERR_CORRUPT; break; }
      word_i += ((pos - seg_bit0 + 127) / 128) * 4;
      if (word_i > words) { err = EBO_ERR_CORRUPT; break; }
    }
    if (err) break;
    if (rd32(rec + 4) != tl || rd32(rec + 8) != tm || rd32(rec + 12) != to) err = EBO_ERR_CORRUPT;
    /* matches, in row order: copy the reference row.  Whole-batch references name literals;
     * window references are distances and may name an earlier match (already copied) */
    if (err == EBO_OK) {
      uint64_t m = match_i - tm;
      for (int64_t b = 0; b < B && err == EBO_OK; ++b) {
        const uint8_t* bm = in + L.off_bitmap + ((size_t)t * nw + (size_t)(b >> 5)) * 4;
        if (!((rd32(bm) >> (b & 31)) & 1u)) continue;
        uint32_t r;
        if (window > 0) {
          const uint32_t dist = in[L.off_refs + m];
          if (dist == 0 || dist > window || (int64_t)dist > b) { err = EBO_ERR_CORRUPT; break; }
          r = (uint32_t)(b - dist);
        } else {
          r = ref_bytes == 2 ? rd16(in + L.off_refs + m * 2) : rd32(in + L.off_refs + m * 4);
        }
        ++m;
        const uint8_t* bmr = in + L.off_bitmap + ((size_t)t * nw + (size_t)(r >> 5)) * 4;
        if ((int64_t)r >= b || (window == 0 && ((rd32(bmr) >> (r & 31)) & 1u))) { err = EBO_ERR_CORRUPT; break; }
        memcpy(sym + ((size_t)t * B + b) * D, sym + ((size_t)t * B + r) * D, (size_t)D * 2);
        memcpy(xhat + ((size_t)b * T + t) * D, xhat + ((size_t)r * T + t) * D, (size_t)D * 4);
      }
    }
  }
  if (err == EBO_OK && (chunk_i != n_chunks || match_i != n_match || out_i != n_out ||
                        word_i != words || lit_total != n_lit))
    err = EBO_ERR_CORRUPT;
  if (err == EBO_OK && sym_out) memcpy(sym_out, sym, N * 2);
  free(sym);
  return err;
}

/* Homogenization Index, [DLRM-EBLC] §III-C Eq. (1): the share of a table's
 * distinct original vectors that quantization merges away,
 * eta = (N_original - N_compressed) / N_original.  0 when every original
 * pattern stays distinct, close to 1 when all collapse into one.  (Tables
 * III and IV print N_compressed / N_original, i.e. 1 - eta.)  N_original = 0
 * gives 0. */
double ebo_homo_index(uint64_t n_original, uint64_t n_compressed) {
  if (n_original == 0) return 0.0;
  return ((double)n_original - (double)n_compressed) / (double)n_original;
}

/* Theoretical speed-up of compressing the traffic, [DLRM-EBLC] §III-D Eq. (2):
 * 1 / (1/CR + B (1/Tc + 1/Td)) with CR the compression ratio, B the network
 * bandwidth and Tc, Td the compression and decompression throughputs (B, Tc,
 * Td in the same unit).  A non-positive CR, Tc or Td gives 0. */
double ebo_speedup(double cr, double bw, double tc, double td) {
  if (!(cr > 0.0) || !(tc > 0.0) || !(td > 0.0) || bw < 0.0) return 0.0;
  return 1.0 / (1.0 / cr + bw * (1.0 / tc + 1.0 / td));
}

/* Offline compressor selection (§III-D "Selection Between Two Encoders"):
 * for each table t, the candidate m (of M) with the largest Eq. (2) speed-up
 * from its sampled ratio cr[t*M + m] and the candidates' throughputs tc[m],
 * td[m]; ties go to the lower index.  Writes choice[t]. */
int ebo_select_modes(const double* cr, const double* tc, const double* td, double bw, int T, int M,
                     uint8_t* choice) {
  if (T < 0 || M < 1 || M > 255 || (T > 0 && (!cr || !tc || !td || !choice))) return EBO_ERR_INVALID_ARG;
  for (int t = 0; t < T; ++t) {
    int best = 0;
    double bs = ebo_speedup(cr[(size_t)t * M], bw, tc[0], td[0]);
    for (int m = 1; m < M; ++m) {
      const double s = ebo_speedup(cr[(size_t)t * M + m], bw, tc[m], td[m]);
      if (s > bs) { bs = s; best = m; }
    }
    choice[t] = (uint8_t)best;
  }
  return EBO_OK;
}
