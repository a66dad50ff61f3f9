/*
 * ebc_oracle.h -- plain, single-threaded CPU oracle of the error-bounded
 * embedding codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this code; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no source with the CUDA path: the container
 * format is implemented here a second time, from its written specification.
 *
 * Method: "Accelerating Communication in Deep Learning Recommendation Model
 * Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
 * cited below as [DLRM-EBLC] with the section / equation / figure.
 *
 * Parity pins (tests/test_oracle_*.py) cover every function here; none is
 * "parity unpinned".
 */
#ifndef EBC_ORACLE_H
#define EBC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EBO_OK 0
#define EBO_ERR_INVALID_ARG 1
#define EBO_ERR_CAPACITY 2
#define EBO_ERR_CORRUPT 3

/* Per-call counts reported by ebo_compress. */
typedef struct {
  uint64_t n_literal;   /* vectors coded through the entropy stream      */
  uint64_t n_match;     /* vectors coded as a back-reference              */
  uint64_t n_outlier;   /* raw values stored (literal vectors only)       */
  uint64_t n_chunks;    /* entries of the chunk-length index              */
  uint64_t bitstream_bytes;
  uint64_t total_bytes;
} ebo_info;

/* Quantization encoder, [DLRM-EBLC] §III-D ("quantization encoder"), with no
 * predictor (§III-B observation 1, "false prediction").  Writes sym[i] in
 * 1..255 for a bin, 0 for an outlier (raw bits kept by the caller).  Returns
 * the number of outliers, or -1 on an invalid bound. */
int64_t ebo_quantize(const float* x, int64_t n, float eb, uint8_t* sym);

/* Dequantization of one symbol (inverse of ebo_quantize for sym != 0). */
float ebo_dequantize(int sym, float eb);

/* 32-bit token hash of one quantized vector (dedup key). */
uint32_t ebo_vector_hash(const uint8_t* sym, const float* x_row, int D);

/* Huffman code lengths for a 256-symbol histogram ([DLRM-EBLC] §III-D,
 * "Optimized Entropy Encoding"), two-queue construction with the length
 * limit lmax.  Returns the number of halving rounds used, -1 on bad args. */
int ebo_huffman_lengths(const uint64_t* freq, int lmax, uint8_t* len);

/* Canonical code values from code lengths (DEFLATE rule). Returns 0, or -1
 * if the lengths violate the Kraft inequality. */
int ebo_canonical_codes(const uint8_t* len, int lmax, uint32_t* code);

/* Iteration-wise decay factor, [DLRM-EBLC] §III-C (OnlineDecay) and §IV-B
 * (Fig. 10). fn: 0 none, 1 linear, 2 stepwise, 3 drop, 4 logarithmic. */
double ebo_decay_factor(int fn, int64_t iter, double m0, int64_t phase_len, int n_steps);

/* Worst-case container size. */
uint64_t ebo_compress_bound(int64_t B, int T, int D);

/* Whole compressor: x is [B,T,D] row-major fp32, eb[T] absolute bounds.
 * Writes the container to out (capacity cap bytes).  Also fills, when the
 * pointers are not NULL: sym_out [T][B][D] quantization codes, ref_out [T][B]
 * (reference vector index for matches, b itself for literals), and
 * lens_out [T][256] code lengths. */
int ebo_compress(const float* x, int64_t B, int T, int D, const float* eb,
                 uint8_t* out, uint64_t cap, ebo_info* info,
                 uint8_t* sym_out, uint32_t* ref_out, uint8_t* lens_out);

/* Per-table coding modes (bit flags; mode 0 is the default pipeline):
 *   EBO_MODE_NO_DEDUP   no vector dedup: every vector of the table is a literal
 *   EBO_MODE_RAW_CODES  no Huffman: every code is stored in 8 bits (all code
 *                       lengths 8, so the canonical code of symbol s is s)
 * Together they give the four per-table choices of the hybrid selection
 * ([DLRM-EBLC] §III-D "Selection Between Two Encoders", Eq. (2)); all of them
 * use the same container. */
#define EBO_MODE_NO_DEDUP 1
#define EBO_MODE_RAW_CODES 2

/* ebo_compress with a mode per table (modes[T] in 0..3, or NULL = all 0). */
int ebo_compress_modes(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes,
                       uint8_t* out, uint64_t cap, ebo_info* info, uint8_t* sym_out, uint32_t* ref_out,
                       uint8_t* lens_out);

/* Sliding-window vector LZ ([DLRM-EBLC] §III-E "extended window size",
 * §IV-D Table VI): with window W in 1..EBO_MAX_WINDOW a vector's reference is
 * the nearest earlier vector of its table within W rows with the same key
 * (a match when codes and raw outlier bits are equal), stored as a one-byte
 * distance; header field 44 holds W (0 = whole-batch first occurrence). */
#define EBO_MAX_WINDOW 255
int ebo_compress_ex(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes, int window,
                    uint8_t* out, uint64_t cap, ebo_info* info, uint8_t* sym_out, uint32_t* ref_out,
                    uint8_t* lens_out);

/* Homogenization Index, [DLRM-EBLC] §III-C Eq. (1). */
double ebo_homo_index(uint64_t n_original, uint64_t n_compressed);

/* Eq. (2) speed-up, [DLRM-EBLC] §III-D. */
double ebo_speedup(double cr, double bw, double tc, double td);

/* Per-table argmax of the Eq. (2) speed-up over M candidates (cr [T][M],
 * tc[M], td[M]); ties to the lower index. */
int ebo_select_modes(const double* cr, const double* tc, const double* td, double bw, int T, int M,
                     uint8_t* choice);

/* Whole decompressor: writes xhat [B,T,D] and, if not NULL, the decoded
 * quantization codes sym_out [T][B][D] (matched vectors carry their
 * reference's codes; a wide-alphabet container then gives EBO_ERR_INVALID_ARG,
 * its codes need ebo_decompress_r). */
int ebo_decompress(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D,
                   float* xhat, uint8_t* sym_out);

/* Wide alphabet (radius R = 512): bins q in (-512, 512), symbols q + 512 in
 * 1..1023 and 0 for an outlier, kept as 16-bit codes; Huffman over 1024
 * symbols with the same length limit; table records of 16 + 1024 bytes; the
 * header's radius field (offset 24) says which alphabet a container uses.  The
 * dedup key sums over 2-code words.  Raw-code mode stores 10-bit codes.  The
 * pages fix no radius; R = 128 stays the default. */
#define EBO_RADIUS 128
#define EBO_RADIUS_WIDE 512
int64_t ebo_quantize_r(const float* x, int64_t n, float eb, int R, uint16_t* sym);
float ebo_dequantize_r(int sym, float eb, int R);
uint32_t ebo_vector_hash_r(const uint16_t* sym, const float* x_row, int D, int R);
/* Huffman lengths / canonical codes over an alphabet of A <= 1024 symbols. */
int ebo_huffman_lengths_n(const uint64_t* freq, int A, int lmax, uint8_t* len);
int ebo_canonical_codes_n(const uint8_t* len, int A, int lmax, uint32_t* code);
uint64_t ebo_compress_bound_r(int64_t B, int T, int D, int R);
/* ebo_compress_ex with radius R (128 or 512); sym_out is [T][B][D] 16-bit,
 * lens_out [T][2R]. */
int ebo_compress_r(const float* x, int64_t B, int T, int D, const float* eb, const uint8_t* modes, int window,
                   int R, uint8_t* out, uint64_t cap, ebo_info* info, uint16_t* sym_out, uint32_t* ref_out,
                   uint8_t* lens_out);
/* ebo_decompress of either alphabet, with 16-bit codes out. */
int ebo_decompress_r(const uint8_t* in, uint64_t in_bytes, int64_t B, int T, int D,
                     float* xhat, uint16_t* sym_out);

#ifdef __cplusplus
}
#endif
#endif
