/*
 * ebc.h -- C ABI of the GB300 error-bounded embedding codec.
 *
 * The codec compresses the gathered embedding-lookup tensor (forward) or the
 * embedding-gradient tensor (backward) x[B][T][D] (fp32, row-major, element
 * (b,t,d) at ((b*T)+t)*D+d; T tables, batch B, embedding dim D) into one
 * contiguous container, and decompresses it back, so that every element obeys
 * the per-table absolute bound |x - xhat| <= eb[t].
 *
 * Method: "Accelerating Communication in Deep Learning Recommendation Model
 * Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272):
 *   - quantization encoder, no predictor ........ §III-D, §III-B observation 1
 *   - vector-based LZ (whole-vector matches) ..... §III-D, §III-E "fixed pattern length"
 *   - Huffman entropy encoder over the bins ...... §III-D "Optimized Entropy Encoding"
 *   - table-wise and iteration-wise bounds ....... §III-C (Eq. 1, OnlineDecay), §IV-B Fig. 10
 *   - one output buffer, metadata with sizes ..... §III-A stage 2, §III-E "Buffer Optimization"
 *
 * Pipeline (all on the GPU, on the caller's stream):
 *   quantize:  q = round_half_even(x * fl32(1/(2 eb_t))), kept if |q| < R and
 *              |x - fl32(q * 2 eb_t)| <= eb_t in fp32, else an outlier whose raw
 *              32 bits are stored; code sym = q + R (1..2R-1), 0 = outlier.  The
 *              radius R is 128 (8-bit codes) unless ebc_set_radius selects 512.
 *   dedup:     within each table, a vector whose codes (and outlier bits) equal
 *              those of an earlier vector of the batch is a match to the first
 *              occurrence; the others are literals.
 *   entropy:   per table, canonical Huffman code (longest code 24 bits) built on
 *              the GPU from the literal codes' histogram; literal vectors are
 *              written MSB-first into a bitstream with a chunk index.
 *
 * Container (little-endian, every section 16-byte aligned):
 *   header 144 B | T table records (eb, counts, 2R code lengths; 272 B each, 1040 B
 *   with radius 512)
 *   | segment records (16 B each) | match bitmap (T x ceil(B/32) u32)
 *   | chunk bit lengths (u16) | match references (u16 row if B <= 65536, else
 *   u32; one-byte distances when the header's window field, at byte 44, is not
 *   0) | bitstream (u32 words; an outlier's code is followed by its 32 raw bits)
 * A segment is max(32, 8192/D) consecutive batch rows of one table; its bits
 * start on a 128-bit boundary.  A chunk is max(1, 128/D) literal vectors of one
 * segment, decoded by one GPU thread.  ebc_compress_chunked writes one such
 * container per slice of the batch, back to back in one buffer.
 *
 * Supported shapes: 0 <= B <= 16,777,215; 0 <= T <= 1024; D a power of two in
 * [4, 512]; B*T*D <= 2^31 (every bitstream word offset then fits 32 bits).
 * Device pointers must be 16-byte aligned.
 *
 * Ownership: the caller allocates and owns every input and output buffer.  A
 * context owns its device scratch (grown on demand, which synchronises the
 * device) and the error-bound schedule.  A context is not thread safe; use one
 * per host thread.
 *
 * Errors: every call returns an EBC_* code.  The compress and decompress calls
 * are asynchronous: argument errors are returned at once; errors found by the
 * kernels (capacity too small, corrupt input) are recorded in the context and
 * returned by the next ebc_last_device_error() or ebc_get_stats(), which
 * synchronise the stream of the last call.
 */
#ifndef EBC_H
#define EBC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EBC_VERSION 1

enum {
  EBC_OK = 0,
  EBC_ERR_INVALID_ARG = 1,    /* bad shape, pointer, bound or schedule        */
  EBC_ERR_CAPACITY = 2,       /* output buffer smaller than the container     */
  EBC_ERR_CORRUPT = 3,        /* container fails validation                   */
  EBC_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out           */
  EBC_ERR_CUDA = 5,           /* a CUDA runtime call failed                   */
  EBC_ERR_NO_DEVICE = 6,      /* no usable sm_103 device                      */
  EBC_ERR_INTERNAL = 7,       /* an internal invariant failed on the device   */
  EBC_ERR_SCRATCH_LIMIT = 8   /* shape too large for ebc_decompress_noalloc   */
};

/* Iteration-wise decay of the error bound, §III-C "Iteration-wise
 * Configuration" and §IV-B Fig. 10.  factor(i) multiplies the base bound (it
 * does not compound); P = phase_len, S = n_steps, m0 = initial multiplier:
 *   LINEAR    m0 - (m0-1) * i/P
 *   STEPWISE  m0 - (m0-1) * floor(i*S/P)/S     (the method's default)
 *   DROP      m0                              (the "Drop_2x" experiment with m0 = 2)
 *   LOG       m0^(1 - i/P)
 * for 0 <= i < P, and 1 for i >= P, for NONE, or when P <= 0. */
typedef enum {
  EBC_DECAY_NONE = 0,
  EBC_DECAY_LINEAR = 1,
  EBC_DECAY_STEPWISE = 2,
  EBC_DECAY_DROP = 3,
  EBC_DECAY_LOG = 4
} ebc_decay;

typedef struct ebc_ctx ebc_ctx;

/* Counts of the last completed compress call of a context. */
typedef struct {
  uint64_t in_bytes;        /* 4*B*T*D                                  */
  uint64_t out_bytes;       /* container bytes                          */
  uint64_t n_vectors;       /* B*T                                      */
  uint64_t n_literal;       /* vectors entropy-coded                    */
  uint64_t n_match;         /* vectors coded as a reference             */
  uint64_t n_outlier;       /* raw values stored                        */
  uint64_t n_chunks;        /* chunk-index entries                      */
  uint64_t bitstream_bytes; /* bytes of the Huffman bitstream section   */
} ebc_stats;

/* Library version (EBC_VERSION). */
int ebc_version(void);

/* Human-readable text of an EBC_* code; never NULL. */
const char* ebc_strerror(int code);

/* Options of a context, fixed when it is created (NULL = the defaults,
 * EBC_CONFIG_DEFAULT).  The paper ("Accelerating Communication in Deep
 * Learning Recommendation Model Training with Dual-Level Adaptive Lossy
 * Compression", §III-D) names the quantization encoder, the vector-based LZ
 * and the Huffman encoder but fixes none of their numbers; this container
 * format fixes two of them (the header records both), and a config that asks
 * for other values is refused with EBC_ERR_INVALID_ARG:
 *   radius         quantization radius: EBC_RADIUS (128; 0 selects it) or
 *                  EBC_RADIUS_WIDE (512), as ebc_set_radius
 *   chunk_vectors  literal vectors per chunk (the decoder's unit of
 *                  parallelism): 0 = the format's max(1, 128/D); nothing else
 *   max_code_len   longest Huffman code: 0 or 24 (the format's); nothing else
 *   dedup          1: vector-based LZ (the default); 0: every vector a literal,
 *                  as EBC_MODE_HUFFMAN for every table (per-table modes set
 *                  later still apply on top)
 *   window         dedup window in rows: 0 = the whole batch, first occurrence
 *                  (the default), 1..255 = nearest earlier vector (ebc_set_window)
 * The radius and window can be changed later with ebc_set_radius and
 * ebc_set_window. */
typedef struct {
  int radius;
  int chunk_vectors;
  int max_code_len;
  int dedup;
  int window;
} ebc_config;
#define EBC_CONFIG_DEFAULT {128, 0, 24, 1, 0}

/* A codec context ([EBLC] §III-E "Compressor Fine-tuning": the compressor's
 * settings are fixed per context, §III-C: so is the bound schedule).
 * Create a context on CUDA device `device` (must be sm_103) with options cfg
 * (host struct, read during the call; NULL = EBC_CONFIG_DEFAULT).  *out
 * receives the context; it is released with ebc_destroy.  Returns
 * EBC_ERR_INVALID_ARG for a bad cfg (checked first, without touching a
 * device), EBC_ERR_NO_DEVICE if the device is absent or not sm_103. */
int ebc_create(ebc_ctx** out, const ebc_config* cfg, int device);

/* Release a context and its device scratch (synchronises the device).  NULL
 * is accepted. */
void ebc_destroy(ebc_ctx* ctx);

/* Table-wise and iteration-wise bounds, §III-C: stores base bounds eb_base[T]
 * (host array, absolute, each finite and > 0) and the schedule; the bound used
 * by ebc_compress(eb = NULL) is fl32(eb_base[t] * factor(iteration)) with the
 * factor computed in double.  Host-only; no device work. */
int ebc_set_error_bounds(ebc_ctx* ctx, const float* eb_base, int T, int64_t iteration,
                         int decay_fn, double m0, int64_t phase_len, int n_steps);

/* Copy the current scheduled bounds (T of them) into eb_out (host). */
int ebc_get_error_bounds(const ebc_ctx* ctx, float* eb_out, int T);

/* [EBLC] §III-A "Training Pipeline with Compression" (the sending buffer is
 * sized before the variable-size output is known).
 * Worst-case container bytes for a [B,T,D] input coded with options cfg
 * (NULL = EBC_CONFIG_DEFAULT; only its radius changes the bound); 0 for an
 * unsupported shape or a bad cfg.  Host-only. */
uint64_t ebc_compress_bound(int64_t B, int T, int D, const ebc_config* cfg);

/* Alphabet of the quantization codes.  Radius 128 (the default): bins q in
 * (-128, 128), 8-bit codes q + 128, 256 symbols.  Radius 512, the wide
 * alphabet: bins q in (-512, 512), codes q + 512 kept as 16 bits in the code
 * scratch, Huffman over 1024 symbols (same 24-bit length limit), table records
 * of 16 + 1024 bytes, 10-bit codes in raw-code mode; values up to 4x farther
 * from zero stop being outliers (32 raw bits each), at twice the scratch and
 * larger tables.  The paper (§III-D) fixes no radius.  The container's
 * radius field (header offset 24) records it. */
#define EBC_RADIUS 128
#define EBC_RADIUS_WIDE 512

/* The radius of this context's later compress and decompress calls (chunked
 * ones too): EBC_RADIUS or EBC_RADIUS_WIDE, else EBC_ERR_INVALID_ARG.  A
 * container of the other alphabet is rejected by the decoder with
 * EBC_ERR_INVALID_ARG (like a container of another shape).
 * ebc_decompress_noalloc decodes radius-128 containers only. */
int ebc_set_radius(ebc_ctx* ctx, int radius);

/* ebc_compress_bound for either radius (0 for another value). */
uint64_t ebc_compress_bound_radius(int64_t B, int T, int D, int radius);

/* The compressor of [EBLC] §III-A "Training Pipeline with Compression" (before
 * the all-to-all) with the hybrid design of §III-D: quantization encoder
 * (no predictor, §III-B observation 1), vector-based LZ, Huffman encoder.
 * Compress d_x[B][T][D] (device, fp32) with bounds eb[T] (host array; NULL =
 * the context's schedule) into d_out (device, out_capacity bytes).  The
 * container size is written to *d_out_bytes (device u64) by the kernels, also
 * when it exceeds out_capacity (then nothing beyond the fixed-size head of the
 * container is written and the context records EBC_ERR_CAPACITY).  `stream` is
 * a cudaStream_t (NULL = legacy default stream).  Asynchronous: returns after
 * the kernels are enqueued.  The input must not be modified until the stream
 * reaches the end of the call. */
int ebc_compress(ebc_ctx* ctx, const float* d_x, int64_t B, int T, int D, const float* eb,
                 void* d_out, uint64_t out_capacity, uint64_t* d_out_bytes, void* stream);

/* ebc_compress for bf16 input (the pages' "mixed precision" embeddings,
 * §IV): d_x[B][T][D] holds bf16 values as their raw 16 bits.  Each value is
 * coded as its exact fp32 value (an outlier keeps those 32 bits), so the
 * container equals ebc_compress of the fp32-converted tensor, while the input
 * read is half as large.  Requires D >= 8 (EBC_ERR_INVALID_ARG otherwise);
 * ebc_decompress returns fp32. */
int ebc_compress_bf16(ebc_ctx* ctx, const uint16_t* d_x, int64_t B, int T, int D, const float* eb,
                      void* d_out, uint64_t out_capacity, uint64_t* d_out_bytes, void* stream);

/* The decompressor of [EBLC] §III-A (after the all-to-all): the inverse of
 * §III-D's encoders, chunk-parallel as in §III-E "Buffer Optimization" /
 * Fig. 7 (bottom).
 * Decompress a container (device, in_bytes bytes) made for the same B, T, D
 * into d_xhat[B][T][D] (device, fp32).  Asynchronous.  A container that fails
 * validation makes the kernels stop without writing out of bounds and records
 * EBC_ERR_CORRUPT (EBC_ERR_INVALID_ARG if its B, T, D differ from the
 * arguments); d_xhat is then unspecified. */
int ebc_decompress(ebc_ctx* ctx, const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B,
                   int T, int D, void* stream);

/* Chunked sending buffer (§III-E "Buffer Optimization", Fig. 7; §IV-D,
 * Fig. 15): the batch is split into n_chunks slices, one per destination rank
 * of the all-to-all, and every slice is coded as a container of its own, all
 * of them in one pass of the kernels and back to back in one buffer.  Slice r
 * holds rows [r*q + min(r, m), (r+1)*q + min(r+1, m)) of the batch, q = B /
 * n_chunks, m = B % n_chunks (the first m slices have one row more; numpy's
 * array_split); a slice may be empty when n_chunks > B.  Dedup, code tables
 * and bitstreams are per slice: container r is exactly what ebc_compress
 * makes of slice r alone, and ebc_decompress restores that slice from it.
 * 1 <= n_chunks <= EBC_MAX_CHUNKS. */
#define EBC_MAX_CHUNKS 256

/* Worst-case bytes of the chunked buffer: the sum of ebc_compress_bound_radius
 * over the slices (0 for an unsupported shape, chunk count or radius). */
uint64_t ebc_compress_chunked_bound(int64_t B, int T, int D, int n_chunks, int radius);

/* Compress d_x[B][T][D] (device, fp32) as n_chunks containers into d_out
 * (device, 16-byte aligned, out_capacity bytes).  The kernels write the
 * container boundaries to d_offsets[0 .. n_chunks] (device u64, caller-owned):
 * container r spans [d_offsets[r], d_offsets[r+1]), every offset a multiple of
 * 16, d_offsets[n_chunks] the total, written also when it exceeds
 * out_capacity (then the containers are not written and the context records
 * EBC_ERR_CAPACITY).  The sizes d_offsets[r+1] - d_offsets[r] are the send
 * counts of an all-to-all, ready on the device without a host round trip.
 * Other arguments and errors as for ebc_compress; the schedule, window and
 * table modes of the context apply to every slice.  Asynchronous. */
int ebc_compress_chunked(ebc_ctx* ctx, const float* d_x, int64_t B, int T, int D, const float* eb,
                         int n_chunks, void* d_out, uint64_t out_capacity, uint64_t* d_offsets,
                         void* stream);
/* The same for bf16 input (see ebc_compress_bf16; D >= 8). */
int ebc_compress_chunked_bf16(ebc_ctx* ctx, const uint16_t* d_x, int64_t B, int T, int D,
                              const float* eb, int n_chunks, void* d_out, uint64_t out_capacity,
                              uint64_t* d_offsets, void* stream);

/* Decompress n_chunks containers from d_in (device, in_bytes bytes, 16-byte
 * aligned) into the rows of their slices in d_xhat[B][T][D] (Fig. 7, bottom:
 * all containers decoded in one pass of the kernels).  d_offsets[0 ..
 * n_chunks] (device u64) are the container boundaries, as written by
 * ebc_compress_chunked or gathered by an all-to-all: each must be a multiple
 * of 16, non-decreasing, and at most in_bytes; container r must hold slice r
 * of the same B, T, D and all containers the same window.  Errors as for
 * ebc_decompress (a bad boundary is EBC_ERR_CORRUPT).  Asynchronous. */
int ebc_decompress_chunked(ebc_ctx* ctx, const void* d_in, uint64_t in_bytes, const uint64_t* d_offsets,
                           int n_chunks, float* d_xhat, int64_t B, int T, int D, void* stream);

/* The receiving side of the all-to-all (Fig. 7, bottom): a container of T
 * tables (from one sender) restores columns [t_off, t_off + T) of d_xhat[B]
 * [T_out][D] (device, fp32, 16-byte aligned); the other columns are not
 * touched.  One call per sender, each on its own stream (with its own context)
 * to decode them in parallel.  0 <= t_off, t_off + T <= T_out, and [B, T_out, D]
 * must be a supported shape, else EBC_ERR_INVALID_ARG.  Otherwise as
 * ebc_decompress. */
int ebc_decompress_columns(ebc_ctx* ctx, const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B, int T,
                           int D, int T_out, int t_off, void* stream);

/* Host-buffer variants (synchronous): the input is copied from host memory
 * h_x (pinned memory is fastest) to context-owned device buffers, processed,
 * and the result copied back.  ebc_compress_host writes the container to
 * h_out (out_capacity bytes) and its size to *out_bytes; it returns
 * EBC_ERR_CAPACITY (with *out_bytes = required size) when it does not fit.
 * ebc_decompress_host reads in_bytes from h_in and writes h_xhat[B][T][D]. */
int ebc_compress_host(ebc_ctx* ctx, const float* h_x, int64_t B, int T, int D, const float* eb,
                      void* h_out, uint64_t out_capacity, uint64_t* out_bytes, void* stream);
int ebc_decompress_host(ebc_ctx* ctx, const void* h_in, uint64_t in_bytes, float* h_xhat,
                        int64_t B, int T, int D, void* stream);

/* Sliding-window vector LZ (the pages' "extended window size" of §III-E,
 * evaluated in §IV-D Table VI).  With window W in 1..255, the following
 * compress calls of the context take as a vector's reference the nearest
 * earlier vector of its table within W rows that has the same key (a match
 * when its codes and raw outlier bits are equal, else a literal), stored as a
 * one-byte distance; references may then chain, and ebc_decompress resolves
 * the chains.  W = 0 (the default) is the whole-batch first occurrence.
 * Returns EBC_ERR_INVALID_ARG for W outside 0..255. */
int ebc_set_window(ebc_ctx* ctx, int window);

/* ---- Per-table hybrid coding (the pages' "Selection Between Two Encoders",
 * §III-D, Eq. (2)) and the Homogenization Index (§III-C, Eq. (1)) ----
 *
 * Every table can be coded in one of four modes; all of them produce the same
 * container, which ebc_decompress reads unchanged:
 *   EBC_MODE_DEDUP_HUFFMAN  vector dedup + per-table canonical Huffman (default)
 *   EBC_MODE_HUFFMAN        no dedup: every vector a literal, Huffman codes
 *   EBC_MODE_DEDUP_RAW      vector dedup, each code stored in 8 bits
 *   EBC_MODE_RAW            no dedup, 8-bit codes
 * The quantization (and so the reconstruction) is the same in every mode. */
typedef enum {
  EBC_MODE_DEDUP_HUFFMAN = 0,
  EBC_MODE_HUFFMAN = 1,
  EBC_MODE_DEDUP_RAW = 2,
  EBC_MODE_RAW = 3
} ebc_mode;

/* Sets the modes (host array modes[T], values 0..3) used by the following
 * compress calls of the context, which must then have this T (else
 * EBC_ERR_INVALID_ARG).  modes == NULL or T == 0 restores mode 0 for every
 * table and any T.  Synchronises the device before it replaces the modes. */
int ebc_set_table_modes(ebc_ctx* ctx, const uint8_t* modes, int T);

/* Per-table counts of the last compress call (synchronises its stream). */
typedef struct {
  uint64_t n_literal;     /* distinct quantized vectors kept (N_compressed of Eq. (1)) */
  uint64_t n_match;       /* vectors coded as references                               */
  uint64_t n_outlier;     /* raw values stored                                         */
  uint64_t n_chunks;      /* chunk-index entries                                       */
  uint64_t payload_bits;  /* bits of the literal codes and outlier values              */
} ebc_table_stats;

/* Writes out[T] for the last compress call, whose T it must be.  Returns the
 * device error recorded by the context, if any (as ebc_last_device_error). */
int ebc_get_table_stats(ebc_ctx* ctx, ebc_table_stats* out, int T);

/* Eq. (1): eta = (N_original - N_compressed) / N_original (0 when
 * N_original = 0): 0 when quantization merges no distinct vectors, towards 1
 * when they collapse into one.  (The pages' Tables III and IV print
 * N_compressed / N_original = 1 - eta.) */
double ebc_homo_index(uint64_t n_original, uint64_t n_compressed);

/* Eq. (2): speed-up = 1 / (1/CR + bw * (1/Tc + 1/Td)), CR the compression
 * ratio, bw the network bandwidth, Tc and Td the compression and
 * decompression throughputs (bw, Tc, Td in one unit).  0 for CR, Tc or Td not
 * positive or bw negative. */
double ebc_speedup(double cr, double bw, double tc, double td);

/* For each table t, the candidate m < M with the largest Eq. (2) speed-up from
 * cr[t*M + m], tc[m], td[m] (ties to the lower m), written to choice[t]. */
int ebc_select_modes(const double* cr, const double* tc, const double* td, double bw, int T, int M,
                     uint8_t* choice);

/* Offline selection on a sample batch (device x[B][T][D], host eb[T], both as
 * for ebc_compress): compresses and decompresses it in each of the four modes
 * (timed with CUDA events on `stream`), takes each table's compression ratio
 * (4*B*D over its payload, chunk-index, reference and record bytes) and each
 * mode's throughputs, and writes the Eq. (2) choice for bandwidth bw (bytes/s)
 * to modes_out[T].  The context's own modes are kept.  Synchronous. */
int ebc_select_table_modes(ebc_ctx* ctx, const float* d_x, int64_t B, int T, int D, const float* eb, double bw,
                           uint8_t* modes_out, void* stream);

/* Eq. (1) per table for a batch: N_compressed = distinct quantized vectors
 * under eb[t] (mode 0), N_original = distinct vectors of the raw values
 * (compressed at the smallest admissible bound, where every value of
 * magnitude above about 3e-36 is an outlier kept bit-exactly).  Writes
 * eta_out[T].  The context's own modes are kept.  Synchronous. */
int ebc_table_homo_index(ebc_ctx* ctx, const float* d_x, int64_t B, int T, int D, const float* eb,
                         double* eta_out, void* stream);

/* Allocation-free decompression.  The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory while they
 * decode -- a process that has handed its device memory to another allocator
 * (where cudaMalloc fails or fragments that pool), or a latency-bound loop in
 * which cudaMalloc/cudaFree would synchronise the device and stall other
 * streams.  It needs no context and allocates nothing: it decodes with the
 * same kernels and gives the same result as ebc_decompress, with their
 * scratch in one static 16 MiB device array of this library (held by every GPU
 * that loads the library until the process exits).
 *
 * Arguments as ebc_decompress; the caller owns d_in and d_xhat.  It works on
 * the current device.  Its first call on a device sets up that device (checks
 * for sm_103 and looks up the array's device address) and should come before
 * any stream capture.  Synchronous: it enqueues the decode on `stream`, waits
 * for the stream, and returns EBC_OK or the decoder's error (EBC_ERR_CORRUPT,
 * EBC_ERR_INVALID_ARG for a container of another shape, EBC_ERR_INTERNAL).
 * Host-side errors: EBC_ERR_INVALID_ARG (bad shape or pointer),
 * EBC_ERR_NO_DEVICE (the current device is not sm_103), EBC_ERR_CUDA, and
 * EBC_ERR_SCRATCH_LIMIT when the shape's scratch does not fit the 16 MiB,
 * in which case nothing is launched.  The scratch is about 4*B*T + 16*T bytes
 * (the row-source table of windowed containers and per-table counters, with
 * the containers' checked layouts, after a 256-byte status block);
 * [8192, 26, 128] needs about 0.85 MB, and shapes of up to about 4 M rows B*T
 * fit.
 * Every call shares the one array per device, and each call clears its status
 * block and counters first: calls whose work overlaps on the GPU (from several host
 * threads, or on several streams) race and must be serialised by the caller. */
int ebc_decompress_noalloc(const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B, int T, int D,
                           void* stream);

/* Counts of the last compress call of the context, read on `stream` (a
 * cudaStream_t; NULL = the stream of the context's last call) after that call
 * has completed; synchronises both streams.  Returns the recorded device error
 * of the context, if any, as ebc_last_device_error. */
int ebc_get_stats(ebc_ctx* ctx, ebc_stats* out, void* stream);

/* Synchronise the stream of the last call and return (and clear) the first
 * error the kernels recorded since the previous query: EBC_OK,
 * EBC_ERR_CAPACITY, EBC_ERR_CORRUPT, EBC_ERR_INVALID_ARG or EBC_ERR_INTERNAL. */
int ebc_last_device_error(ebc_ctx* ctx);

/* Failure-detection test aid.  Every device-side wait of the codec is bounded:
 * the quantize kernel polls the barrier of each input tile at most 2^22 times,
 * and a wait that runs out records EBC_ERR_DEVICE_TIMEOUT, drains the tile
 * copies still in flight (waiting for them with the full limit), and stops its
 * block; the kernels after it then write nothing to the output, and the next
 * ebc_last_device_error() returns the code.  This sets the number of polls of
 * the FIRST tile wait of each quantize block of the following compress calls
 * (0 <= polls <= 2^22; a negative value restores the full limit, which is the
 * default).  With 0 the first wait gives up before looking, so a test can run
 * the time-out path without hanging anything; later waits keep the full
 * limit.  Host-only; EBC_ERR_INVALID_ARG for a null context or polls > 2^22. */
int ebc_set_first_wait_polls(ebc_ctx* ctx, int polls);

/* Per-kernel timing (tracing aid).  While enabled, every kernel launch of the
 * context is bracketed by a pair of CUDA events on its stream (up to 2048
 * launches between reads).  ebc_get_profile synchronises on the last event,
 * writes one entry per kernel name (launch count and summed milliseconds) into
 * out[capacity], sets *count, and clears the record. */
typedef struct {
  char name[32];
  uint64_t launches;
  double total_ms;
} ebc_kernel_time;

int ebc_set_profiling(ebc_ctx* ctx, int enable);
int ebc_get_profile(ebc_ctx* ctx, ebc_kernel_time* out, int capacity, int* count);

#ifdef __cplusplus
}
#endif
#endif /* EBC_H */
