// ebc_decompress.cu -- decompression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (Huffman and vector-based LZ decoding, dequantization) and §III-E
// ("parallel decompression" of chunks).  Three launches:
//   k_dec_prep     every CTA checks the header and layout; the first T CTAs
//                  build each table's canonical decode tables (2^11-entry
//                  first-level table + long codes); the others, one warp per
//                  segment, check the segment records against each other and
//                  write one descriptor per chunk (start bit, length, rows)
//   k_dec_chunks   one thread per chunk: decodes its literal rows (codes,
//                  inline outliers) and writes them straight to the output
//   k_dec_matches  copies each matched row from its (literal) reference
// Every read of the container is bounds-checked; a failed check records
// EBC_ERR_CORRUPT and stops the remaining work without out-of-bounds access.
#include <cstdint>

#include "ebc_internal.cuh"

namespace ebc {

__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ unsigned long long ld64(const uint8_t* p) {
  return *reinterpret_cast<const unsigned long long*>(p);
}
__device__ __forceinline__ unsigned long long dpad16(unsigned long long n) { return (n + 15ull) & ~15ull; }

__device__ __forceinline__ void dec_fail(Glob* g, uint32_t epoch, int code) {
  atomicExch(&g->dstat, status_word(epoch, code));
  record_error(g, code);
}

__device__ __forceinline__ bool dec_aborted(const Glob* g, uint32_t epoch) {
  const unsigned int st = __ldcg(&g->dstat);
  return (st >> 8) == (epoch & 0xFFFFFFu) && (st & 0xFFu) != 0u;
}

__device__ __forceinline__ bool eb_usable(float eb) {
  if (!(eb >= 1.17549435e-38f) || !(eb <= 3.40282347e+38f)) return false;
  const float ebx2 = __fmul_rn(2.0f, eb);
  if (!(ebx2 <= 3.40282347e+38f)) return false;
  return __fdiv_rn(1.0f, ebx2) >= 1.17549435e-38f;
}

struct Layout {
  unsigned long long n_lit, n_match, n_out, n_chunks, words;
  unsigned long long off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;
};

// Header checks (h: the 144 header bytes in shared memory).  Returns an EBC_*
// code; on success *L holds the section layout recomputed from the counts.
__device__ int parse_header(const uint8_t* h, unsigned long long in_bytes, const Shape& sh, Layout* L) {
  const int T = sh.T;
  const unsigned long long nvec = (unsigned long long)sh.B * (unsigned long long)T;
  if (in_bytes < kHeaderBytes) return EBC_ERR_CORRUPT;
  if (ld32(h) != kMagic || ld32(h + 4) != kFormatVersion) return EBC_ERR_CORRUPT;
  if (ld64(h + 8) != (unsigned long long)sh.B || ld32(h + 16) != (uint32_t)T || ld32(h + 20) != (uint32_t)sh.D)
    return EBC_ERR_INVALID_ARG;
  if (ld32(h + 24) != (uint32_t)kRadius || ld32(h + 28) != (uint32_t)kLmax || ld32(h + 32) != (uint32_t)sh.SB ||
      ld32(h + 36) != (uint32_t)sh.KC || ld32(h + 40) != (uint32_t)sh.ref_bytes || ld32(h + 44) != 0u)
    return EBC_ERR_CORRUPT;
  L->n_lit = ld64(h + 48);
  L->n_match = ld64(h + 56);
  L->n_out = ld64(h + 64);
  L->n_chunks = ld64(h + 72);
  L->words = ld64(h + 80);
  if (L->n_lit + L->n_match != nvec || L->n_lit > nvec || L->n_chunks > nvec ||
      L->n_out > nvec * (unsigned long long)sh.D || L->words > (1ull << 34))
    return EBC_ERR_CORRUPT;
  L->off_seg = kHeaderBytes + (unsigned long long)T * kTableRecBytes;
  L->off_bitmap = L->off_seg + (unsigned long long)T * sh.nseg * kSegRecBytes;
  L->off_chunks = L->off_bitmap + dpad16((unsigned long long)T * sh.nw * 4ull);
  L->off_refs = L->off_chunks + dpad16(L->n_chunks * 2ull);
  L->off_bits = L->off_refs + dpad16(L->n_match * (unsigned long long)sh.ref_bytes);
  L->total = L->off_bits + L->words * 4ull;
  if (ld64(h + 88) != L->off_seg || ld64(h + 96) != L->off_bitmap || ld64(h + 104) != L->off_chunks ||
      ld64(h + 112) != L->off_refs || ld64(h + 120) != L->off_bits || ld64(h + 128) != L->total ||
      ld64(h + 136) != 0ull || L->total > in_bytes)
    return EBC_ERR_CORRUPT;
  return EBC_OK;
}

// Exclusive scan of v across one warp.
__device__ __forceinline__ uint32_t warp_excl(uint32_t v, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += n;
  }
  *total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - v;
}

// ---------------------------------------------------------------------------
// k_dec_prep: grid T + ceil(T * nseg / 8), 256 threads.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_dec_prep(const uint8_t* __restrict__ in, unsigned long long in_bytes,
                                                   Shape sh, Work w, uint32_t epoch) {
  using G = Geo<D>;
  __shared__ __align__(16) uint8_t s_hdr[kHeaderBytes];
  __shared__ Layout s_L;
  __shared__ int s_code;
  __shared__ uint8_t s_len[256];
  __shared__ uint32_t s_count[kLmax + 2], s_next[kLmax + 2], s_offset[kLmax + 2];
  __shared__ int s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = sh.T;
  Glob* g = w.glob;
  if (in_bytes >= kHeaderBytes && tid < (int)(kHeaderBytes / 16))
    reinterpret_cast<uint4*>(s_hdr)[tid] = reinterpret_cast<const uint4*>(in)[tid];
  __syncthreads();
  if (tid == 0) {
    s_code = parse_header(s_hdr, in_bytes, sh, &s_L);
    s_bad = 0;
    if (blockIdx.x == 0) {
      if (s_code != EBC_OK) {
        dec_fail(g, epoch, s_code);
      } else {
        g->n_lit = s_L.n_lit; g->n_match = s_L.n_match; g->n_out = s_L.n_out; g->n_chunks = s_L.n_chunks;
        g->words = s_L.words; g->off_seg = s_L.off_seg; g->off_bitmap = s_L.off_bitmap;
        g->off_chunks = s_L.off_chunks; g->off_refs = s_L.off_refs; g->off_bits = s_L.off_bits;
        g->total = s_L.total;
      }
    }
  }
  __syncthreads();
  if (s_code != EBC_OK) return;
  const Layout L = s_L;

  if ((int)blockIdx.x < T) {
    // ---- decode tables of table t ----
    const int t = blockIdx.x;
    const uint8_t* rec = in + kHeaderBytes + (size_t)t * kTableRecBytes;
    const uint32_t len = rec[16 + tid];
    s_len[tid] = (uint8_t)len;
    if (tid < kLmax + 2) s_count[tid] = 0;
    __syncthreads();
    if (len > (uint32_t)kLmax) s_bad = 1;
    else if (len) atomicAdd(&s_count[len], 1u);
    __syncthreads();
    if (tid == 0) {
      const float eb = __uint_as_float(ld32(rec));
      unsigned long long kraft = 0;
      for (int l = 1; l <= kLmax; ++l) kraft += (unsigned long long)s_count[l] << (kLmax - l);
      if (kraft > (1ull << kLmax) || !eb_usable(eb)) s_bad = 1;
      uint32_t c = 0, off = 0;
      s_count[0] = 0;
      for (int l = 1; l <= kLmax; ++l) {
        c = (c + s_count[l - 1]) << 1;
        s_next[l] = c;
        s_offset[l] = off;
        off += s_count[l];
      }
      DecTab* dt = w.dtab + t;
      dt->ebx2 = __fmul_rn(2.0f, eb);
      for (int l = 0; l <= kLmax; ++l) {
        dt->first[l] = l ? s_next[l] : 0u;
        dt->count[l] = l ? s_count[l] : 0u;
        dt->offset[l] = l ? s_offset[l] : 0u;
      }
    }
    __syncthreads();
    if (s_bad) {
      if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
      return;
    }
    uint16_t* lut = w.lut + (size_t)t * (1u << kLutBits);
    for (int i = tid; i < (1 << kLutBits); i += 256) lut[i] = 0;
    __syncthreads();
    if (len) {
      uint32_t rank = 0;
      for (int j = 0; j < tid; ++j) rank += (s_len[j] == len);
      const uint32_t code = s_next[len] + rank;
      w.dtab[t].sorted[s_offset[len] + rank] = (uint8_t)tid;
      if (len <= (uint32_t)kLutBits) {
        const uint32_t lo = code << (kLutBits - len), n = 1u << (kLutBits - len);
        for (uint32_t i = 0; i < n; ++i) lut[lo + i] = (uint16_t)(tid | (len << 8));
      }
    }
    return;
  }

  // ---- one warp per segment: literal rows and chunk descriptors ----
  const int nsegT = T * sh.nseg;
  const int seg = ((int)blockIdx.x - T) * 8 + warp;
  if (seg >= nsegT) return;
  const int t = seg / sh.nseg;
  const int s = seg - t * sh.nseg;
  const int64_t B = sh.B;
  const int64_t row0 = (int64_t)s * G::kSB;
  const uint32_t* rec = reinterpret_cast<const uint32_t*>(in + L.off_seg) + 4ull * seg;
  const uint32_t word_off = rec[0], chunk_base = rec[1], match_base = rec[2], nbits = rec[3];
  unsigned long long nx_word, nx_chunk, nx_match;
  if (seg + 1 < nsegT) {
    nx_word = rec[4];
    nx_chunk = rec[5];
    nx_match = rec[6];
  } else {
    nx_word = L.words;
    nx_chunk = L.n_chunks;
    nx_match = L.n_match;
  }
  const uint32_t* bmt = reinterpret_cast<const uint32_t*>(in + L.off_bitmap) + (size_t)t * sh.nw;
  // literal rows, in row order: words 0..31 on the lanes, then words 32..63
  uint32_t nlit = 0, nvalid_rows = 0;
  uint16_t* litrow = w.litrow + (size_t)seg * G::kSB;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int wi = half * 32 + lane;
    uint32_t litw = 0, valid = 0;
    if (wi < G::kBmWords) {
      const int64_t gw = (int64_t)s * G::kBmWords + wi;
      if (gw < sh.nw) {
        const int64_t nv = B - (row0 + (int64_t)wi * 32);
        valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
        const uint32_t bm = bmt[gw];
        if (bm & ~valid) s_bad = 1;             // match bits past the batch
        litw = ~bm & valid;
      }
    }
    uint32_t tot;
    uint32_t k = nlit + warp_excl(__popc(litw), &tot);
    uint32_t vt;
    warp_excl(__popc(valid), &vt);
    nlit += tot;
    nvalid_rows += vt;
    for (uint32_t m = litw; m; m &= m - 1) litrow[k++] = (uint16_t)(wi * 32 + __ffs(m) - 1);
  }
  const uint32_t nmatch = nvalid_rows - nlit;
  const uint32_t nchunks = (nlit + G::kKC - 1) / G::kKC;
  const unsigned long long seg_words = ((nbits + 127ull) >> 7) * 4ull;
  bool ok = (unsigned long long)chunk_base + nchunks == nx_chunk && nx_chunk <= L.n_chunks &&
            (unsigned long long)match_base + nmatch == nx_match && nx_match <= L.n_match &&
            (unsigned long long)word_off + seg_words == nx_word && nx_word <= L.words &&
            (seg != 0 || (word_off == 0 && chunk_base == 0 && match_base == 0));
  // chunk start bits
  uint32_t cstart = 0;
  if (ok) {
    const uint16_t* cl = reinterpret_cast<const uint16_t*>(in + L.off_chunks) + chunk_base;
    uint32_t acc = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t c = half * 32 + lane;
      const uint32_t len = c < nchunks ? (uint32_t)cl[c] : 0u;
      uint32_t tot;
      const uint32_t st = acc + warp_excl(len, &tot);
      if (c < nchunks) {
        const unsigned long long start = (unsigned long long)word_off * 32ull + st;
        const uint32_t rows = min((uint32_t)G::kKC, nlit - c * G::kKC);
        w.cdesc[chunk_base + c] = make_uint4((uint32_t)start, (uint32_t)(start >> 32) | (len << 16), (uint32_t)seg,
                                             (c * G::kKC) | (rows << 16));
      }
      acc += tot;
    }
    cstart = acc;
    ok = cstart == nbits;
  }
  if (!__all_sync(0xffffffffu, ok) || s_bad) {
    if (lane == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
  }
}

// ---------------------------------------------------------------------------
// k_dec_chunks: one thread per chunk (grid-stride).  The thread decodes its
// chunk's codes with the first-level table (long codes by the canonical
// first-code search), reads the 32 raw bits after each outlier code, and
// writes each literal row with 16-byte stores.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_dec_chunks(const uint8_t* __restrict__ in, Shape sh, Work w,
                                                     float* __restrict__ xhat, uint32_t epoch) {
  using G = Geo<D>;
  Glob* g = w.glob;
  if (dec_aborted(g, epoch)) return;
  const unsigned long long n_chunks = __ldcg(&g->n_chunks), n_words = __ldcg(&g->words);
  const unsigned long long off_bits = __ldcg(&g->off_bits);
  const uint32_t* words = reinterpret_cast<const uint32_t*>(in + off_bits);
  const int T = sh.T;
  const int nsegT = T * sh.nseg;
  for (unsigned long long j = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; j < n_chunks;
       j += (unsigned long long)gridDim.x * blockDim.x) {
    const uint4 dsc = __ldcg(&w.cdesc[j]);
    const unsigned long long start = (unsigned long long)dsc.x | ((unsigned long long)(dsc.y & 0xffffu) << 32);
    const uint32_t clen = dsc.y >> 16;
    const int seg = (int)dsc.z;
    const uint32_t first = dsc.w & 0xffffu, rows = dsc.w >> 16;
    if (seg >= nsegT || rows == 0u || first + rows > (uint32_t)G::kSB || start + clen > n_words * 32ull) {
      dec_fail(g, epoch, EBC_ERR_CORRUPT);
      continue;
    }
    const int t = seg / sh.nseg;
    const int s = seg - t * sh.nseg;
    const uint16_t* lut = w.lut + (size_t)t * (1u << kLutBits);
    const DecTab* dt = w.dtab + t;
    const float ebx2 = __ldg(&dt->ebx2);
    const unsigned long long wlim = (start + clen + 31ull) >> 5;
    unsigned long long wp = start >> 5;
    auto ldw = [&](unsigned long long i) -> unsigned long long {
      return i < wlim ? (unsigned long long)__ldg(words + i) : 0ull;
    };
    unsigned long long buf = (ldw(wp) << 32) | ldw(wp + 1);
    const uint32_t skip = (uint32_t)(start & 31ull);
    buf <<= skip;
    int nb = 64 - (int)skip;
    wp += 2;
    uint32_t used = 0;
    bool bad = false;
    const uint16_t* lrow = w.litrow + (size_t)seg * G::kSB + first;
    for (uint32_t k = 0; k < rows && !bad; ++k) {
      const int64_t b = (int64_t)s * G::kSB + lrow[k];
      float4* dst = reinterpret_cast<float4*>(xhat + ((size_t)b * T + t) * D);
      for (int q4 = 0; q4 < D / 4; ++q4) {
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (nb < 32) {
            buf |= ldw(wp++) << (32 - nb);
            nb += 32;
          }
          const uint32_t e = __ldg(lut + (uint32_t)(buf >> (64 - kLutBits)));
          uint32_t len = e >> 8, sym = e & 0xffu;
          if (len == 0u) {
            for (int l = kLutBits + 1; l <= kLmax; ++l) {
              const uint32_t code = (uint32_t)(buf >> (64 - l));
              const uint32_t f = __ldg(&dt->first[l]);
              if (code - f < __ldg(&dt->count[l])) {
                sym = __ldg(&dt->sorted[__ldg(&dt->offset[l]) + code - f]);
                len = (uint32_t)l;
                break;
              }
            }
            if (len == 0u) {
              bad = true;
              len = 1;
            }
          }
          buf <<= len;
          nb -= (int)len;
          used += len;
          if (sym == 0u) {
            if (nb < 32) {
              buf |= ldw(wp++) << (32 - nb);
              nb += 32;
            }
            o[q] = __uint_as_float((uint32_t)(buf >> 32));
            buf <<= 32;
            nb -= 32;
            used += 32;
          } else {
            o[q] = __fmul_rn((float)((int)sym - kRadius), ebx2);
          }
        }
        dst[q4] = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    if (bad || used != clen) dec_fail(g, epoch, EBC_ERR_CORRUPT);
  }
}

// ---------------------------------------------------------------------------
// k_dec_matches: one CTA per (table, segment); each matched row copies its
// reference row, which is always an earlier literal of the same table.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_dec_matches(const uint8_t* __restrict__ in, Shape sh, Work w,
                                                      float* __restrict__ xhat, uint32_t epoch) {
  using G = Geo<D>;
  __shared__ uint32_t s_bm[G::kBmWords];
  __shared__ uint32_t s_pre[G::kBmWords + 1];
  __shared__ uint16_t s_mrow[G::kSB];
  __shared__ uint32_t s_mref[G::kSB];
  __shared__ int s_bad;
  Glob* g = w.glob;
  if (dec_aborted(g, epoch)) return;
  const int tid = threadIdx.x;
  const int seg = blockIdx.x;
  const int t = seg / sh.nseg;
  const int s = seg - t * sh.nseg;
  const int64_t B = sh.B;
  const int T = sh.T;
  const int64_t row0 = (int64_t)s * G::kSB;
  const unsigned long long off_seg = __ldcg(&g->off_seg), off_bitmap = __ldcg(&g->off_bitmap);
  const unsigned long long off_refs = __ldcg(&g->off_refs), n_match = __ldcg(&g->n_match);
  const uint32_t match_base = reinterpret_cast<const uint32_t*>(in + off_seg + (unsigned long long)seg * kSegRecBytes)[2];
  const uint32_t* bmt = reinterpret_cast<const uint32_t*>(in + off_bitmap) + (size_t)t * sh.nw;
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    s_bm[tid] = wi < sh.nw ? bmt[wi] : 0u;
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (tid < 32) {   // prefix of match counts over the segment's bitmap words (<= 64)
    const uint32_t a = tid * 2 < G::kBmWords ? __popc(s_bm[tid * 2]) : 0u;
    const uint32_t c = tid * 2 + 1 < G::kBmWords ? __popc(s_bm[tid * 2 + 1]) : 0u;
    uint32_t tot;
    const uint32_t ex = warp_excl(a + c, &tot);
    if (tid * 2 < G::kBmWords) s_pre[tid * 2] = ex;
    if (tid * 2 + 1 < G::kBmWords) s_pre[tid * 2 + 1] = ex + a;
    if (tid == 0) s_pre[G::kBmWords] = tot;
  }
  __syncthreads();
  const uint32_t nm = s_pre[G::kBmWords];
  if ((unsigned long long)match_base + nm > n_match) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  // references: one thread per matched row, loads in parallel
  const uint8_t* refs = in + off_refs;
  for (int r = tid; r < G::kSB; r += 256) {
    const int64_t b = row0 + r;
    if (b >= B || !((s_bm[r >> 5] >> (r & 31)) & 1u)) continue;
    const uint32_t rank = s_pre[r >> 5] + __popc(s_bm[r >> 5] & ((1u << (r & 31)) - 1u));
    const unsigned long long mi = (unsigned long long)match_base + rank;
    const uint32_t ref = sh.ref_bytes == 2 ? (uint32_t)reinterpret_cast<const uint16_t*>(refs)[mi]
                                           : reinterpret_cast<const uint32_t*>(refs)[mi];
    if ((int64_t)ref >= b || ((bmt[ref >> 5] >> (ref & 31)) & 1u)) s_bad = 1;
    s_mrow[rank] = (uint16_t)r;
    s_mref[rank] = ref;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  // copy: flat over (matched row, float4), four independent copies in flight per thread
  constexpr int kQ = D / 4;
  const uint32_t n4 = nm * kQ;
  for (uint32_t i0 = tid; i0 < n4; i0 += 4 * 256) {
    float4 v[4];
    size_t dst[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t i = i0 + k * 256;
      if (i < n4) {
        const uint32_t m = i / kQ, q = i % kQ;
        const int64_t b = row0 + s_mrow[m];
        v[k] = *reinterpret_cast<const float4*>(xhat + ((size_t)s_mref[m] * T + t) * D + 4 * q);
        dst[k] = ((size_t)b * T + t) * D + 4 * q;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (i0 + k * 256 < n4) __stcs(reinterpret_cast<float4*>(xhat + dst[k]), v[k]);
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D>
static void launch_decompress_d(const uint8_t* in, unsigned long long in_bytes, const Shape& sh, const Work& w,
                                float* xhat, uint32_t epoch, cudaStream_t st, Prof* prof) {
  const unsigned nsegT = (unsigned)(sh.T * sh.nseg);
  prof_begin(prof, "k_dec_prep", st);
  k_dec_prep<D><<<(sh.T > 0 ? sh.T : 1) + (nsegT + 7) / 8, 256, 0, st>>>(in, in_bytes, sh, w, epoch);
  prof_end(prof, st);
  if (nsegT) {
    const unsigned long long max_chunks = (unsigned long long)nsegT * Geo<D>::kChunks;
    unsigned grid = (unsigned)((max_chunks + 255) / 256);
    const unsigned cap = (unsigned)(sh.nsm > 0 ? sh.nsm : 152) * 8u;
    if (grid > cap) grid = cap;
    prof_begin(prof, "k_dec_chunks", st);
    k_dec_chunks<D><<<grid, 256, 0, st>>>(in, sh, w, xhat, epoch);
    prof_end(prof, st);
    prof_begin(prof, "k_dec_matches", st);
    k_dec_matches<D><<<nsegT, 256, 0, st>>>(in, sh, w, xhat, epoch);
    prof_end(prof, st);
  }
}

cudaError_t launch_decompress(const uint8_t* in, unsigned long long in_bytes, const Shape& sh, const Work& w,
                              float* xhat, uint32_t epoch, cudaStream_t st, Prof* prof) {
  switch (sh.D) {
    case 4: launch_decompress_d<4>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 8: launch_decompress_d<8>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 16: launch_decompress_d<16>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 32: launch_decompress_d<32>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 64: launch_decompress_d<64>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 128: launch_decompress_d<128>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 256: launch_decompress_d<256>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    case 512: launch_decompress_d<512>(in, in_bytes, sh, w, xhat, epoch, st, prof); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ebc
