// ebc_internal.cuh -- types, format constants and device helpers shared by the
// codec's CUDA kernels (sm_103a).  See include/ebc.h for the container format.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ebc.h"

namespace ebc {

// ---- container format, version 2 ----
constexpr int kRadius = 128;               // codes q + 128 for |q| < 128; 0 = outlier
constexpr int kRadiusWide = 512;           // the wide alphabet: codes q + 512 for |q| < 512, 16-bit
constexpr int kMaxSyms = 1024;
constexpr int kLmax = 24;                  // longest Huffman code
constexpr uint32_t kMagic = 0x31434245u;   // "EBC1"
constexpr uint32_t kFormatVersion = 2;
constexpr uint32_t kHeaderBytes = 144;
constexpr uint32_t kTableRecBytes = 272;   // f32 eb, u32 n_lit, n_match, n_out, u8 len[256]
                                           // (16 + 1024 bytes with the wide alphabet)
constexpr uint32_t kSegRecBytes = 16;      // u32 word_off, chunk_base, match_base, n_bits
constexpr int kMaxT = 1024;
constexpr int kMaxB = 16777215;

// ---- decoder ----
constexpr int kLutBits = 11;               // first-level decode table: 2^11 entries

constexpr unsigned long long kEmptySlot = ~0ull;

constexpr int kWaitLimit = 1 << 22;        // polls of an mbarrier before a wait gives up

// Shape-derived constants of one call.
//
// The batch may be split into R slices (the rows of one destination rank of an
// all-to-all each), every slice coded as a container of its own.  The first
// B % R slices hold B / R + 1 rows, the others B / R.  The coding unit is one
// table of one slice: unit u = r * T + t, so the units of a container are
// consecutive.  With R = 1 a unit is a table.
struct Shape {
  int64_t B;
  int T;
  int D;
  int SB;         // rows per segment: max(32, 8192 / D)
  int KC;         // literal rows per chunk: max(1, 128 / D)
  int nseg;       // segments per unit: ceil(Bc / SB)
  int nw;         // bitmap words per unit: ceil(Bc / 32)
  uint32_t S;     // dedup slots per unit (power of two >= 2 Bc, >= 64)
  int ref_bytes;  // 1 with a window (distances), else 2 if B <= 65536 else 4 (of the R = 1 container)
  int nsm;        // SMs of the device (grid sizing)
  uint64_t symstride;  // bytes per table in the code scratch: B*D rounded up to 16
  int window;     // dedup window in rows (0 = whole batch, first occurrence; else nearest earlier, 1..255)
  int fold;       // 1: segment offsets are built per unit inside k_codebook (nseg <= kFoldMaxSeg);
                  // 0: by k_layout, per 8-segment tile
  int R;          // slices of the batch (containers)
  int U;          // units: R * T
  int64_t Bq;     // B / R
  int Brem;       // B % R
  int64_t Bc;     // rows of the largest slice
  int qseg;       // quantization segments per table: ceil(B / SB) (k_quantize works on whole tables)
  int W;          // bytes per code in the scratch: 1 (radius 128) or 2 (radius 512)
  int A;          // symbols of the alphabet: 256 or 1024
  int first_wait; // polls of each quantize CTA's first input-tile wait (a test aid; normally the full limit)
  int T_out;      // decode: tables of the output rows (T, or more when decoding into columns)
  int t_off;      // decode: output column of the container's first table
};

// The two alphabets, by code width W in bytes.
template <int W>
struct Alph {
  static constexpr int kR = W == 1 ? kRadius : kRadiusWide;   // radius: codes q + R for |q| < R
  static constexpr int kA = 2 * kR;                             // symbols (0 = outlier)
  static constexpr int kRawLen = W == 1 ? 8 : 10;               // bits of a raw code (log2 kA)
  static constexpr int kLenShift = W == 1 ? 8 : 10;             // decode-table entry: sym | len << shift
  static constexpr uint32_t kRecBytes = 16u + (uint32_t)kA;     // table record
};
__host__ __device__ inline uint32_t table_rec_bytes(int A) { return 16u + (uint32_t)A; }

// Codes of four consecutive elements (one lane's share): one word of four
// 8-bit codes, or two words of two 16-bit codes (code of element k in byte /
// half-word k, little-endian).
template <int W>
struct QuadOf;
template <>
struct QuadOf<1> {
  using T = uint32_t;
};
template <>
struct QuadOf<2> {
  using T = uint2;
};
__device__ __forceinline__ uint32_t quad_code(uint32_t v, int q) { return (v >> (8 * q)) & 0xffu; }
__device__ __forceinline__ uint32_t quad_code(uint2 v, int q) {
  return ((q < 2 ? v.x : v.y) >> (16 * (q & 1))) & 0xffffu;
}
__device__ __forceinline__ bool quad_eq(uint32_t a, uint32_t b) { return a == b; }
__device__ __forceinline__ bool quad_eq(uint2 a, uint2 b) { return a.x == b.x && a.y == b.y; }
// a zero code (an outlier) among the four
__device__ __forceinline__ bool quad_has_zero(uint32_t v) { return ((v - 0x01010101u) & ~v & 0x80808080u) != 0u; }
__device__ __forceinline__ bool quad_has_zero(uint2 v) {
  return (((v.x - 0x00010001u) & ~v.x & 0x80008000u) | ((v.y - 0x00010001u) & ~v.y & 0x80008000u)) != 0u;
}

constexpr int kFoldMaxSeg = 256;
constexpr int kMaxWindow = 255;
constexpr int kMaxSlices = EBC_MAX_CHUNKS;

// Rows of slice r: [slice_row0, slice_row0 + slice_rows).
__host__ __device__ inline int64_t slice_row0(const Shape& sh, int r) {
  return (int64_t)r * sh.Bq + (r < sh.Brem ? r : sh.Brem);
}
__host__ __device__ inline int64_t slice_rows(const Shape& sh, int r) { return sh.Bq + (r < sh.Brem ? 1 : 0); }
// The slice holding batch row b (0 <= b < B).
__host__ __device__ inline int slice_of_row(const Shape& sh, int64_t b) {
  if (sh.R == 1) return 0;
  const int64_t big = (int64_t)sh.Brem * (sh.Bq + 1);   // rows of the longer slices
  return b < big ? (int)(b / (sh.Bq + 1)) : sh.Brem + (int)((b - big) / sh.Bq);
}
// Bytes per reference of a container of n rows.
__host__ __device__ inline int ref_bytes_of(int64_t n, int window) { return window > 0 ? 1 : (n <= 65536 ? 2 : 4); }
__host__ __device__ inline int div_up(int64_t a, int b) { return (int)((a + b - 1) / b); }

// Section layout of one container, relative to its first byte (base).
struct ContLay {
  unsigned long long n_lit, n_match, n_out, n_chunks, words;
  unsigned long long base, off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;
  uint32_t word0, chunk0, match0;   // bitstream words, chunks and matches of the units before the container
  uint32_t ref_bytes;
};

// Section layout of one container as the decoder checks it (offsets relative to base).
struct Layout {
  unsigned long long n_lit, n_match, n_out, n_chunks, words;
  unsigned long long off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;
  unsigned long long base;          // the container's first byte in the input
  unsigned long long row0, n;       // the batch rows it restores: [row0, row0 + n)
  unsigned int window, ref_bytes;   // dedup window (0 = whole batch) and bytes per reference
  unsigned int nseg, nw;            // segments and bitmap words per table
};

// Per-table coding modes (bit flags; 0 = vector dedup + Huffman codes).
constexpr uint32_t kModeNoDedup = 1;   // every vector of the table is a literal
constexpr uint32_t kModeRawCodes = 2;  // every code 8 bits (lengths all 8: code of symbol s is s)

// Per-table absolute bounds of one compress call, passed by value.
struct EbParams {
  float eb[kMaxT];
};

// Device-resident state of a context.
struct Glob {
  unsigned int done;      // arrival counter of the last-block reductions
  unsigned int cstat;     // (epoch << 8) | status of the last compress
  unsigned int dstat;     // (epoch << 8) | status of the last decompress
  unsigned int sticky;    // first device error since the last query (0 = none)
  unsigned int window;    // the window of the container being decoded (0 = whole batch)
  unsigned int cabort;    // (epoch << 8) | status: a compress call given up by its quantize kernel
  unsigned int pad[2];
  unsigned long long n_lit, n_match, n_out, n_chunks, words;
  unsigned long long off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;
};

// Device scratch of a context.  Sizes follow Shape.
struct Work {
  const uint8_t* modes;        // [T] per-table modes, or null (all 0)
  uint32_t mode_or;            // modes added to every table's (dedup switched off for the context)
  unsigned long long* tab_bits;   // [U] bits of the unit's literal codes and outlier values
  // compress
  uint8_t* sym;                // [T][B][D] quantization codes (W bytes each), table t at t * symstride
                               //   (16-byte aligned)
  uint32_t* vhash;             // [T][B] dedup key
  unsigned long long* slots;   // [U][S] (hash << 32 | first row); all ones = empty
  uint32_t* bitmap;            // [U][nw] match bits (rows of the unit's slice)
  uint32_t* ref;               // [T][B] reference row (batch row) of matched rows
  uint32_t* seg_hist;          // [U*nseg][A] literal code histogram per segment
  uint4* seg_cnt;              // [U*nseg] {literals, matches, outliers, chunks}
  uint4* seg_desc;             // [groups] totals {words, chunks, matches} of each group of segments
  uint4* tile_base;            // [groups] absolute base of each group
  uint4* seg_base;             // [U*nseg] {words, chunks, matches} relative to its group, and the bit count
                               // (a group: the unit when Shape::fold, else 8 consecutive segments)
  uint32_t* tab_hist;          // [U][A] literal code histogram per unit
  uint4* tab_cnt;              // [U] {literals, matches, outliers, chunks}
  uint4* tab_rec;              // [U] the first 16 bytes of the unit's table record: eb, literals, matches, outliers
  uint32_t* tabcode;           // [U][A] code << 8 | length
  ContLay* cont;               // [R] container layouts
  // decompress
  uint4* uacc;                 // [U] per-unit accumulators {literals, matches, outliers, arrived CTAs}, zero
                               //   between calls (the last CTA of each unit empties its own)
  uint2* cacc;                 // [R] per-container accumulators {outliers, arrived units}, zero between calls
  Layout* lay;                 // [R] each container's section layout, as the decoder's header check found it
  uint32_t* srcrow;            // [T][B] windowed containers: each row's source row (itself for a literal)
  Glob* glob;
};

// The modes of table t in a compress call.
__device__ __forceinline__ uint32_t table_mode(const Work& w, int t) {
  return (w.modes ? (uint32_t)w.modes[t] : 0u) | w.mode_or;
}

// Error bits kept in Glob::sticky / status words.
__host__ __device__ constexpr unsigned int status_word(uint32_t epoch, int code) {
  return (epoch << 8) | (unsigned int)code;
}

// ---- small device helpers ----
__device__ __forceinline__ uint32_t lowbias32(uint32_t v) {
  // C. Wellons' 32-bit integer mixer "lowbias32" (hash-prospector).
  v ^= v >> 16;
  v *= 0x7feb352dU;
  v ^= v >> 15;
  v *= 0x846ca68bU;
  v ^= v >> 16;
  return v;
}

__device__ __forceinline__ void record_error(Glob* g, int code) {
  atomicCAS(&g->sticky, 0u, (unsigned int)code);
}

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  // read-once input: evict-first streaming load
  return __ldcs(reinterpret_cast<const float4*>(p));
}

template <int D>
struct Geo {
  static constexpr int kSB = (8192 / D) < 32 ? 32 : (8192 / D);   // rows per segment
  static constexpr int kKC = (128 / D) < 1 ? 1 : (128 / D);       // rows per chunk
  static constexpr int kLPR = D / 4 < 32 ? D / 4 : 32;            // lanes per row
  static constexpr int kRPS = 32 / kLPR;                          // rows per 128-element slab
  static constexpr int kSPR = D / 128 < 1 ? 1 : D / 128;          // slabs per row
  static constexpr int kSlabs = kSB * D / 128;                    // slabs per segment
  static constexpr int kSlabsPerWarp = kSlabs / 8;                // 8 warps per CTA
  static constexpr int kRowsPerWarp = kSB / 8;
  static constexpr int kBmWords = kSB / 32;                       // bitmap words per segment
  static constexpr int kChunks = kSB / kKC;                       // max chunks per segment
  static constexpr int kSegSyms = kSB * D;
};

// Ascending bitonic sort of n (a power of two) keys in shared memory by the
// whole CTA; every thread takes its share of the pairs of each stage.
__device__ inline void bitonic_sort_smem(unsigned long long* key, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = key[i], b = key[l];
          if ((a > b) == ((i & k) == 0)) {
            key[i] = b;
            key[l] = a;
          }
        }
      }
      __syncthreads();
    }
}

// Exclusive scan of one uint4 per thread over the CTA (s_warp: 8 slots).
__device__ __forceinline__ uint4 add4(uint4 a, uint4 b) {
  return make_uint4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ inline uint4 block_excl_scan4(uint4 v, uint4* total, uint4* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4 inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint4 n;
    n.x = __shfl_up_sync(0xffffffffu, inc.x, off);
    n.y = __shfl_up_sync(0xffffffffu, inc.y, off);
    n.z = __shfl_up_sync(0xffffffffu, inc.z, off);
    n.w = __shfl_up_sync(0xffffffffu, inc.w, off);
    if (lane >= off) inc = add4(inc, n);
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  uint4 pre = make_uint4(0, 0, 0, 0), tot = make_uint4(0, 0, 0, 0);
  const int nwarps = blockDim.x >> 5;
  for (int i = 0; i < nwarps; ++i) {
    if (i < warp) pre = add4(pre, s_warp[i]);
    tot = add4(tot, s_warp[i]);
  }
  __syncthreads();
  *total = tot;
  return make_uint4(pre.x + inc.x - v.x, pre.y + inc.y - v.y, pre.z + inc.z - v.z, pre.w + inc.w - v.w);
}

// Ascending bitonic sort of one 64-bit key per thread over a 256-thread CTA:
// partners closer than a warp trade through shuffles, the others through
// shared memory.  Returns the key of rank threadIdx.x.
__device__ __forceinline__ unsigned long long bitonic_sort256(unsigned long long v, unsigned long long* s_key) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 2; k <= 256; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      unsigned long long p;
      if (j >= 32) {
        s_key[tid] = v;
        __syncthreads();
        p = s_key[tid ^ j];
        __syncthreads();
      } else {
        p = __shfl_xor_sync(0xffffffffu, v, j);
      }
      const bool up = (tid & k) == 0;        // this run ascends
      const bool low = (tid & j) == 0;       // lower element of the pair
      const unsigned long long mn = v < p ? v : p, mx = v < p ? p : v;
      v = (up == low) ? mn : mx;
    }
  }
  return v;
}

// Sorts the keys of the symbols in use, ascending, into s_key[0 .. n): each
// thread passes its kPer keys (~0 = not in use).  The used keys are compacted
// by a CTA scan; up to 256 of them are sorted in registers and shuffles, more
// by a shared-memory sort of all of them.  Returns n.
template <int kPer>
__device__ int sort_used_keys(const unsigned long long (&key)[kPer], unsigned long long* s_key, uint4* s_warp) {
  const int tid = threadIdx.x;
  uint32_t mine = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) mine += key[k] != ~0ull;
  uint4 tot;
  const uint32_t at = block_excl_scan4(make_uint4(mine, 0, 0, 0), &tot, s_warp).x;
  const int n = (int)tot.x;
  uint32_t p = at;
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (key[k] != ~0ull) s_key[p++] = key[k];
  if (n > 256)
    for (int i = n + tid; i < kPer * 256; i += 256) s_key[i] = ~0ull;
  __syncthreads();
  if (n <= 256) {
    const unsigned long long v = tid < n ? s_key[tid] : ~0ull;
    __syncthreads();   // s_key becomes the sort's scratch
    const unsigned long long sk = bitonic_sort256(v, s_key);
    __syncthreads();
    s_key[tid] = sk;
    __syncthreads();
  } else {
    bitonic_sort_smem(s_key, kPer * 256);
  }
  return n;
}

// Canonical ranks over a 256-thread CTA: thread tid holds the code lengths of
// symbols k * 256 + tid (k < kPer); rank[k] is the number of symbols of the
// same length with a smaller index (in its warp from a match mask, in the
// warps and rounds before from counts).  s_wcnt: 8 x (kLmax + 1) words,
// s_run: kLmax + 1 words of shared scratch.
template <int kPer>
__device__ void canonical_ranks(const uint32_t (&len)[kPer], uint32_t (&rank)[kPer], uint32_t* s_wcnt,
                                uint32_t* s_run) {
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  constexpr int kL = kLmax + 1;
  if (tid < kL) s_run[tid] = 0u;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    for (int i = tid; i < 8 * kL; i += 256) s_wcnt[i] = 0u;
    __syncthreads();
    const unsigned same = __match_any_sync(0xffffffffu, len[k]);
    if (lane == __ffs(same) - 1) s_wcnt[wp * kL + len[k]] = (uint32_t)__popc(same);
    __syncthreads();
    uint32_t r = s_run[len[k]] + (uint32_t)__popc(same & ((1u << lane) - 1u));
    for (int j = 0; j < wp; ++j) r += s_wcnt[j * kL + len[k]];
    rank[k] = r;
    __syncthreads();
    if (tid < kL) {
      uint32_t add = 0;
      for (int j = 0; j < 8; ++j) add += s_wcnt[j * kL + tid];
      s_run[tid] += add;
    }
    __syncthreads();   // the counts are read before the next round clears them
  }
}

// ---- programmatic dependent launch ----
// Every kernel of a call is launched with programmatic stream serialization.
// On entry it lets the next kernel of the stream launch (which happens once
// all of its own CTAs have started, so the next grid fills the SMs its tail
// frees), then waits until the kernels before it have completed and their
// memory is visible, before it reads anything they wrote.  A kernel whose
// predecessor is not a kernel waits for nothing.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- optional per-kernel timing (host side, defined with the C ABI) ----
struct Prof;
void prof_begin(Prof* p, const char* name, cudaStream_t st);
void prof_end(Prof* p, cudaStream_t st);

// ---- launchers (one per direction; D is dispatched to the templated kernels) ----
// out_bytes: the total size; chunk_off: null, or [R] the first byte of each container.
cudaError_t launch_compress(const void* x, bool bf16, const Shape& sh, const EbParams& ep, const Work& w,
                            uint8_t* out, unsigned long long cap, unsigned long long* out_bytes,
                            unsigned long long* chunk_off, uint32_t epoch, cudaStream_t st, Prof* prof);
// offs: null (one container of in_bytes), or [R + 1] container boundaries in device memory.
cudaError_t launch_decompress(const uint8_t* in, unsigned long long in_bytes, const unsigned long long* offs,
                              const Shape& sh, const Work& w, float* xhat, uint32_t epoch, cudaStream_t st,
                              Prof* prof);
cudaError_t set_kernel_attributes();
cudaError_t set_decoder_attributes();

}  // namespace ebc
