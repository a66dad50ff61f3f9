// ebc_decompress.cu -- decompression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (Huffman and vector-based LZ decoding, dequantization) and §III-E
// ("parallel decompression" of chunks; one or several containers, one per
// batch slice, decoded in the same pass).  The unit is a table of one
// container.  Three launches:
//   k_dec_prep     every CTA checks every header and layout; the first U CTAs
//                  build each unit's canonical decode tables (2^11-entry
//                  first-level table + long codes); the others, one warp per
//                  segment, check the segment records against each other and
//                  write one descriptor per chunk (start bit, length, rows)
//   k_dec_chunks   one thread per chunk, one CTA per run of 64 chunks (listed
//                  in a run map written by k_dec_prep): decodes its literal
//                  rows (codes, inline outliers) from shared-memory copies of
//                  the bitstream and writes them straight to the output
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
  unsigned long long off_seg, off_bitmap, off_chunks, off_refs, off_bits, total;   // relative to base
  unsigned long long base;          // the container's first byte in the input
  unsigned long long row0, n;       // the batch rows it restores: [row0, row0 + n)
  unsigned int window, ref_bytes;   // dedup window (0 = whole batch) and bytes per reference
  unsigned int nseg, nw;            // segments and bitmap words per table
  unsigned int chunk0, match0;      // chunks and matches of the containers before it
};

// Header checks of a container of n rows and `bytes` bytes (h: its first
// byte).  Returns an EBC_* code; on success *L holds the section layout
// recomputed from the counts.
__device__ int parse_header(const uint8_t* h, unsigned long long bytes, unsigned long long n, const Shape& sh,
                            Layout* L) {
  const int T = sh.T;
  const unsigned long long nvec = n * (unsigned long long)T;
  if (bytes < kHeaderBytes) return EBC_ERR_CORRUPT;
  if (ld32(h) != kMagic || ld32(h + 4) != kFormatVersion) return EBC_ERR_CORRUPT;
  if (ld64(h + 8) != n || ld32(h + 16) != (uint32_t)T || ld32(h + 20) != (uint32_t)sh.D)
    return EBC_ERR_INVALID_ARG;
  const uint32_t radius = ld32(h + 24);   // the alphabet: both are valid, the call decodes one of them
  if (radius != (uint32_t)kRadius && radius != (uint32_t)kRadiusWide) return EBC_ERR_CORRUPT;
  if (radius != (uint32_t)(sh.A / 2)) return EBC_ERR_INVALID_ARG;
  if (ld32(h + 28) != (uint32_t)kLmax || ld32(h + 32) != (uint32_t)sh.SB ||
      ld32(h + 36) != (uint32_t)sh.KC || ld32(h + 44) > (uint32_t)kMaxWindow)
    return EBC_ERR_CORRUPT;
  L->n = n;
  L->nseg = (unsigned int)div_up((int64_t)n, sh.SB);
  L->nw = (unsigned int)div_up((int64_t)n, 32);
  L->window = ld32(h + 44);
  L->ref_bytes = (unsigned int)ref_bytes_of((int64_t)n, (int)L->window);   // windowed: one-byte distances
  if (ld32(h + 40) != L->ref_bytes) return EBC_ERR_CORRUPT;
  L->n_lit = ld64(h + 48);
  L->n_match = ld64(h + 56);
  L->n_out = ld64(h + 64);
  L->n_chunks = ld64(h + 72);
  L->words = ld64(h + 80);
  if (L->n_lit + L->n_match != nvec || L->n_lit > nvec ||
      L->n_chunks > (unsigned long long)T * L->nseg * (unsigned long long)(sh.SB / sh.KC) ||
      L->n_out > nvec * (unsigned long long)sh.D || L->words > (1ull << 34))
    return EBC_ERR_CORRUPT;
  L->off_seg = kHeaderBytes + (unsigned long long)T * table_rec_bytes(sh.A);
  L->off_bitmap = L->off_seg + (unsigned long long)T * L->nseg * kSegRecBytes;
  L->off_chunks = L->off_bitmap + dpad16((unsigned long long)T * L->nw * 4ull);
  L->off_refs = L->off_chunks + dpad16(L->n_chunks * 2ull);
  L->off_bits = L->off_refs + dpad16(L->n_match * (unsigned long long)L->ref_bytes);
  L->total = L->off_bits + L->words * 4ull;
  if (ld64(h + 88) != L->off_seg || ld64(h + 96) != L->off_bitmap || ld64(h + 104) != L->off_chunks ||
      ld64(h + 112) != L->off_refs || ld64(h + 120) != L->off_bits || ld64(h + 128) != L->total ||
      ld64(h + 136) != 0ull || L->total > bytes)
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
// k_dec_prep: grid U + ceil(U * nseg / 8), 256 threads.  Every CTA checks all
// R headers (thread r: container r) and takes the chunk and match bases of
// each container from a scan of their counts; a failed check stops every CTA.
// ---------------------------------------------------------------------------
template <int D, int W>
__global__ void __launch_bounds__(256) k_dec_prep(const uint8_t* __restrict__ in, unsigned long long in_bytes,
                                                   const unsigned long long* __restrict__ offs, Shape sh, Work w,
                                                   uint32_t epoch) {
  pdl_enter();
  using G = Geo<D>;
  constexpr int kA = Alph<W>::kA, kPer = kA / 256;
  __shared__ Layout s_L[8];   // the containers of this CTA's units: r_lo .. r_lo + 7
  __shared__ uint32_t s_nc[kMaxSlices + 1], s_nm[kMaxSlices + 1], s_win[kMaxSlices];
  __shared__ unsigned long long s_tot[4];   // literals, outliers, words, bytes of all containers
  __shared__ int s_code;
  __shared__ uint8_t s_len[kA];
  __shared__ uint32_t s_wcnt[8 * (kLmax + 1)], s_run[kLmax + 1];   // canonical ranks
  __shared__ uint32_t s_count[kLmax + 2], s_next[kLmax + 2], s_offset[kLmax + 2];
  __shared__ int s_bad;
  __shared__ uint32_t s_c0, s_c1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = sh.T;
  const int U = sh.U;
  const int nsegT = U * sh.nseg;
  Glob* g = w.glob;
  // the containers this CTA needs
  int r_lo;
  if ((int)blockIdx.x < U) {
    r_lo = (int)blockIdx.x / T;
  } else {
    const int seg0 = ((int)blockIdx.x - U) * 8;
    r_lo = seg0 < nsegT ? (seg0 / sh.nseg) / T : 0;
  }
  if (tid == 0) {
    s_code = EBC_OK;
    s_bad = 0;
  }
  if (tid < 4) s_tot[tid] = 0ull;
  __syncthreads();
  Layout L{};
  int code = EBC_OK;
  if (tid < sh.R) {
    const unsigned long long lo = offs ? offs[tid] : 0ull, hi = offs ? offs[tid + 1] : in_bytes;
    if ((lo & 15ull) != 0ull || lo > hi || hi > in_bytes) {
      code = EBC_ERR_CORRUPT;
    } else {
      uint4 hdr[kHeaderBytes / 16];   // the header, by independent 16-byte loads
      if (hi - lo >= kHeaderBytes) {
#pragma unroll
        for (int k = 0; k < (int)(kHeaderBytes / 16); ++k) hdr[k] = reinterpret_cast<const uint4*>(in + lo)[k];
      }
      code = parse_header(reinterpret_cast<const uint8_t*>(hdr), hi - lo, (unsigned long long)slice_rows(sh, tid),
                          sh, &L);
      L.base = lo;
      L.row0 = (unsigned long long)slice_row0(sh, tid);
    }
    // counts for the scan (zero for a container that failed: its check stops the decode)
    s_nc[tid] = code == EBC_OK ? (uint32_t)L.n_chunks : 0u;
    s_nm[tid] = code == EBC_OK ? (uint32_t)L.n_match : 0u;
    s_win[tid] = code == EBC_OK ? L.window : 0u;
    if (code != EBC_OK) {
      atomicCAS(&s_code, EBC_OK, code);
    } else if (blockIdx.x == 0) {
      atomicAdd(&s_tot[0], L.n_lit);
      atomicAdd(&s_tot[1], L.n_out);
      atomicAdd(&s_tot[2], L.words);
      atomicAdd(&s_tot[3], L.total);
    }
  }
  __syncthreads();
  if (tid == 0) {   // chunk and match bases of the containers; one window for all of them
    uint32_t c = 0, m = 0;
    for (int r = 0; r < sh.R; ++r) {
      const uint32_t a = s_nc[r], b = s_nm[r];
      s_nc[r] = c;
      s_nm[r] = m;
      c += a;
      m += b;
      if (s_win[r] != s_win[0] && s_code == EBC_OK) s_code = EBC_ERR_CORRUPT;
    }
    s_nc[sh.R] = c;
    s_nm[sh.R] = m;
  }
  __syncthreads();
  if (tid < sh.R && code == EBC_OK) {
    L.chunk0 = s_nc[tid];
    L.match0 = s_nm[tid];
    if (tid >= r_lo && tid < r_lo + 8) s_L[tid - r_lo] = L;
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    if (s_code != EBC_OK) {
      dec_fail(g, epoch, s_code);
    } else {
      g->n_match = s_nm[sh.R];
      g->n_chunks = s_nc[sh.R];
      g->window = s_win[0];
      g->n_lit = s_tot[0];
      g->n_out = s_tot[1];
      g->words = s_tot[2];
      g->total = s_tot[3];
    }
  }
  if (s_code != EBC_OK) return;

  if ((int)blockIdx.x < U) {
    // ---- decode tables of unit u = (slice r, table t) ----
    const int u = blockIdx.x;
    const int t = u % T;
    const Layout Lc = s_L[0];
    const uint8_t* cin = in + Lc.base;
    const uint8_t* rec = cin + kHeaderBytes + (size_t)t * Alph<W>::kRecBytes;
    uint32_t lens[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      lens[k] = rec[16 + k * 256 + tid];
      s_len[k * 256 + tid] = (uint8_t)lens[k];
    }
    if (tid < kLmax + 2) s_count[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (lens[k] > (uint32_t)kLmax) s_bad = 1;
      else if (lens[k]) atomicAdd(&s_count[lens[k]], 1u);
    }
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
      DecTab* dt = w.dtab + u;
      dt->ebx2 = __fmul_rn(2.0f, eb);
      // the unit's chunk range (segment records are checked against each other by the segment warps)
      const uint32_t* srec = reinterpret_cast<const uint32_t*>(cin + Lc.off_seg);
      uint32_t c0 = 0, c1 = 0;
      if (Lc.nseg > 0) {
        c0 = srec[4ull * ((unsigned long long)t * Lc.nseg) + 1];
        c1 = t + 1 < T ? srec[4ull * ((unsigned long long)(t + 1) * Lc.nseg) + 1] : (uint32_t)Lc.n_chunks;
      }
      if (c0 > c1 || c1 > Lc.n_chunks) s_bad = 1;
      c0 += Lc.chunk0;   // over all containers
      c1 += Lc.chunk0;
      if (c1 > dec_max_chunks(sh)) s_bad = 1;
      dt->chunk0 = c0;
      dt->chunk1 = c1;
      dt->t = (uint32_t)t;
      dt->bits_off = Lc.base + Lc.off_bits;
      dt->n_words = Lc.words;
      dt->row0 = Lc.row0;
      s_c0 = c0;
      s_c1 = c1;
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
    {   // this unit's run slots [c0 / kDecRun + u, c1 / kDecRun + u + 1): its runs, then one empty slot at most
      const uint32_t c0 = s_c0, c1 = s_c1;
      const uint32_t lo = c0 / kDecRun + (uint32_t)u, hi = c1 / kDecRun + (uint32_t)u + 1u;
      const uint32_t nruns = (c1 - c0 + kDecRun - 1) / kDecRun;
      for (uint32_t r = lo + tid; r < hi; r += 256) {
        const uint32_t k = r - lo;
        const uint32_t j0 = c0 + k * kDecRun;
        w.runmap[r] = k < nruns ? make_uint4((uint32_t)u, j0, min(j0 + (uint32_t)kDecRun, c1), 0u)
                                : make_uint4(~0u, 0u, 0u, 0u);
      }
    }
    uint16_t* lut = w.lut + (size_t)u * (1u << kLutBits);
    for (int i = tid; i < (1 << kLutBits); i += 256) lut[i] = 0;
    __syncthreads();
    {
      // each symbol's rank among the symbols of its length below it: its index in sorted[] is
      // offset[len] + rank, its code first[len] + rank
      uint32_t rk[kPer];
      canonical_ranks<kPer>(lens, rk, s_wcnt, s_run);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const uint32_t len = lens[k], sy = (uint32_t)(k * 256 + tid);
        if (!len) continue;
        const uint32_t code = s_next[len] + rk[k];
        w.dtab[u].sorted[s_offset[len] + rk[k]] = (uint16_t)sy;
        if (len <= (uint32_t)kLutBits) {
          const uint32_t lo = code << (kLutBits - len), n = 1u << (kLutBits - len);
          for (uint32_t i = 0; i < n; ++i) lut[lo + i] = (uint16_t)(sy | (len << Alph<W>::kLenShift));
        }
      }
    }
    if (Lc.window && Lc.nseg > 0) {
      // window references: every row's source (itself for a literal, b - distance for a match),
      // from the unit's bitmap and one-byte distances, then the chains resolved to their
      // literal roots (pointer jumping, CTA barriers between rounds)
      const int64_t n = (int64_t)Lc.n, row0 = (int64_t)Lc.row0;
      const int64_t nw = Lc.nw;
      const uint32_t* bmt = reinterpret_cast<const uint32_t*>(cin + Lc.off_bitmap) + (size_t)t * nw;
      const uint8_t* dist = cin + Lc.off_refs;
      const uint32_t* srec = reinterpret_cast<const uint32_t*>(cin + Lc.off_seg);
      const unsigned long long mbase = srec[4ull * ((unsigned long long)t * Lc.nseg) + 2];
      uint32_t* src = w.srcrow + (size_t)t * sh.B + row0;
      unsigned long long carry = 0;
      for (int64_t base = 0; base < nw; base += 256) {
        const int64_t wi = base + tid;
        const uint32_t bm = wi < nw ? __ldcg(&bmt[wi]) : 0u;
        // matches before this word: a CTA-wide exclusive scan of the words' counts
        uint32_t wt;
        const uint32_t in_warp = warp_excl((uint32_t)__popc(bm), &wt);
        if (lane == 0) s_count[warp] = wt;
        __syncthreads();
        uint32_t before = 0, all = 0;
        for (int k = 0; k < 8; ++k) {
          if (k < warp) before += s_count[k];
          all += s_count[k];
        }
        __syncthreads();
        const unsigned long long rank0 = mbase + carry + before + in_warp;
        if (wi < nw) {
          for (int j = 0; j < 32; ++j) {
            const int64_t b = wi * 32 + j;   // row of the slice
            if (b >= n) break;
            uint32_t from = (uint32_t)(row0 + b);
            if ((bm >> j) & 1u) {
              const unsigned long long k = rank0 + __popc(bm & ((1u << j) - 1u));
              const uint32_t d = k < Lc.n_match ? dist[k] : 0u;
              if (d == 0u || d > Lc.window || (int64_t)d > b) s_bad = 1;
              else from = (uint32_t)(row0 + b - d);
            }
            src[b] = from;
          }
        }
        carry += all;
      }
      __syncthreads();
      if (s_bad) {
        if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
        return;
      }
      int rounds = 1;
      while ((1ll << rounds) < n) ++rounds;
      for (int rd = 0; rd <= rounds; ++rd) {
        for (int64_t b = tid; b < n; b += 256) {
          const uint32_t s = src[b];
          if (s != (uint32_t)(row0 + b)) {
            const uint32_t s2 = src[s - row0];   // one step further (a literal points at itself)
            if (s2 != s) src[b] = s2;
          }
        }
        __syncthreads();
      }
    }
    return;
  }

  // ---- one warp per segment: literal rows and chunk descriptors ----
  const int seg = ((int)blockIdx.x - U) * 8 + warp;
  if (seg >= nsegT) return;
  const int u = seg / sh.nseg;
  const int s = seg - u * sh.nseg;
  const int r = u / T;
  const int t = u - r * T;
  const Layout Lc = s_L[r - r_lo];
  if (s >= (int)Lc.nseg) return;   // past the end of a shorter slice
  const uint8_t* cin = in + Lc.base;
  const int64_t B = (int64_t)Lc.n;                // rows of the slice
  const int64_t row0 = (int64_t)s * G::kSB;      // within the slice
  const int64_t nw = Lc.nw;
  const unsigned long long ri = (unsigned long long)t * Lc.nseg + s;   // record of the segment
  const uint32_t* rec = reinterpret_cast<const uint32_t*>(cin + Lc.off_seg) + 4ull * ri;
  const uint32_t word_off = rec[0], chunk_base = rec[1], match_base = rec[2], nbits = rec[3];
  unsigned long long nx_word, nx_chunk, nx_match;
  if (ri + 1 < (unsigned long long)T * Lc.nseg) {
    nx_word = rec[4];
    nx_chunk = rec[5];
    nx_match = rec[6];
  } else {
    nx_word = Lc.words;
    nx_chunk = Lc.n_chunks;
    nx_match = Lc.n_match;
  }
  const uint32_t* bmt = reinterpret_cast<const uint32_t*>(cin + Lc.off_bitmap) + (size_t)t * nw;
  // literal rows, in row order: words 0..31 on the lanes, then words 32..63
  uint32_t nlit = 0, nvalid_rows = 0;
  uint16_t* litrow = w.litrow + (size_t)seg * G::kSB;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int wi = half * 32 + lane;
    uint32_t litw = 0, valid = 0;
    if (wi < G::kBmWords) {
      const int64_t gw = (int64_t)s * G::kBmWords + wi;
      if (gw < nw) {
        const int64_t nv = B - (row0 + (int64_t)wi * 32);
        valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
        const uint32_t bm = bmt[gw];
        if (bm & ~valid) s_bad = 1;             // match bits past the slice
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
  bool ok = (unsigned long long)chunk_base + nchunks == nx_chunk && nx_chunk <= Lc.n_chunks &&
            (unsigned long long)match_base + nmatch == nx_match && nx_match <= Lc.n_match &&
            (unsigned long long)word_off + seg_words == nx_word && nx_word <= Lc.words &&
            (ri != 0 || (word_off == 0 && chunk_base == 0 && match_base == 0));
  // chunk start bits
  uint32_t cstart = 0;
  if (ok) {
    const uint16_t* cl = reinterpret_cast<const uint16_t*>(cin + Lc.off_chunks) + chunk_base;
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
        w.cdesc[Lc.chunk0 + chunk_base + c] = make_uint4((uint32_t)start, (uint32_t)(start >> 32) | (len << 16),
                                                         (uint32_t)seg, (c * G::kKC) | (rows << 16));
      }
      acc += tot;
    }
    cstart = acc;
    ok = cstart == nbits;
  }
  // matched rows: {destination, source} row pairs of the batch, in (unit, row) order
  if (__all_sync(0xffffffffu, ok)) {
    const uint8_t* refs = cin + Lc.off_refs;
    const int64_t brow0 = (int64_t)Lc.row0;
    uint32_t mbase = match_base;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int wi = half * 32 + lane;
      uint32_t mw = 0;
      if (wi < G::kBmWords) {
        const int64_t gw = (int64_t)s * G::kBmWords + wi;
        if (gw < nw) mw = bmt[gw];
      }
      uint32_t tot;
      uint32_t k = mbase + warp_excl(__popc(mw), &tot);
      for (uint32_t m = mw; m; m &= m - 1) {
        const int64_t b = row0 + wi * 32 + __ffs(m) - 1;   // row of the slice
        uint32_t ref;
        if (Lc.window) {   // a distance back, within the window; the row there may itself be a match
          const uint32_t dist = refs[k];
          if (dist == 0u || dist > Lc.window || (int64_t)dist > b) {
            ok = false;
            break;
          }
          ref = (uint32_t)(b - dist);
        } else {           // whole slice: the first occurrence, always a literal
          ref = Lc.ref_bytes == 2 ? (uint32_t)reinterpret_cast<const uint16_t*>(refs)[k]
                                  : reinterpret_cast<const uint32_t*>(refs)[k];
          if ((int64_t)ref >= b || ((bmt[ref >> 5] >> (ref & 31)) & 1u)) {
            ok = false;
            break;
          }
        }
        w.mdesc[Lc.match0 + k] = make_uint2((uint32_t)((brow0 + b) * sh.T_out + sh.t_off + t),
                                            (uint32_t)((brow0 + ref) * sh.T_out + sh.t_off + t));
        ++k;
      }
      mbase += tot;
    }
  }
  if (!__all_sync(0xffffffffu, ok) || s_bad) {
    if (lane == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
  }
}

// ---------------------------------------------------------------------------
// k_dec_chunks: one thread per chunk, one CTA per run of kDecRun consecutive
// chunks of one table (the run map lists the runs first, so every CTA with
// work precedes the empty ones).  The run's chunks are consecutive in the
// bitstream: the CTA copies their words into shared memory with coalesced
// loads (when they fit), together with the table's decode tables and the 256
// reconstruction values.  Each thread then decodes its chunk with the
// first-level table (long codes by the canonical first-code search), reads the
// 32 raw bits after each outlier code, and writes each literal row with
// 16-byte stores.
// ---------------------------------------------------------------------------
template <int D>
struct DecStage {
  static constexpr int kWords = D <= 128 ? 4096 : 8192;   // 16 / 32 KiB of bitstream per CTA
};

// Decodes one chunk (rows literal rows of D codes) starting at bit `start`;
// ldw(i) returns word i of the bitstream.  Returns the number of bits read.
template <int D, int W, class LoadWord>
__device__ __forceinline__ unsigned long long decode_chunk(LoadWord ldw, unsigned long long start,
                                                           const uint16_t* s_lut, const float* s_val,
                                                           const uint32_t* s_first, const uint32_t* s_count,
                                                           const uint32_t* s_offset, const uint16_t* s_sorted,
                                                           const uint16_t* lrow, uint32_t rows, int64_t row0, int T,
                                                           int t, float* __restrict__ xhat, bool* bad) {
  // bit window: the next stream bits are w0:w1 from bit `pos` of w0 (pos < 32); w0 is word wp - 2
  unsigned long long wp = start >> 5;
  uint32_t pos = (uint32_t)(start & 31ull);
  uint32_t w0 = ldw(wp), w1 = ldw(wp + 1);
  wp += 2;
  for (uint32_t k = 0; k < rows; ++k) {
    const int64_t b = row0 + lrow[k];
    float4* dst = reinterpret_cast<float4*>(xhat + ((size_t)b * T + t) * D);
#pragma unroll 2
    for (int q4 = 0; q4 < D / 4; ++q4) {
      float o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t peek = __funnelshift_l(w1, w0, pos);   // the next 32 bits
        const uint32_t e = s_lut[peek >> (32 - kLutBits)];
        uint32_t len = e >> Alph<W>::kLenShift, sym = e & ((1u << Alph<W>::kLenShift) - 1u);
        if (len == 0u) {   // a code longer than the first-level table
          for (int l = kLutBits + 1; l <= kLmax; ++l) {
            const uint32_t code = peek >> (32 - l);
            if (code - s_first[l] < s_count[l]) {
              sym = s_sorted[s_offset[l] + code - s_first[l]];
              len = (uint32_t)l;
              break;
            }
          }
          if (len == 0u) {
            *bad = true;
            len = 1;
          }
        }
        pos += len;
        if (pos >= 32u) {
          pos -= 32u;
          w0 = w1;
          w1 = ldw(wp++);
        }
        o[q] = s_val[sym];
        if (sym == 0u) {   // outlier: the next 32 bits are the raw value
          o[q] = __uint_as_float(__funnelshift_l(w1, w0, pos));
          w0 = w1;
          w1 = ldw(wp++);
        }
      }
      dst[q4] = make_float4(o[0], o[1], o[2], o[3]);
    }
  }
  return (wp - 2ull) * 32ull + pos - start;
}

template <int D, int W>
__global__ void __launch_bounds__(kDecRun) k_dec_chunks(const uint8_t* __restrict__ in, Shape sh, Work w,
                                                         float* __restrict__ xhat, uint32_t epoch) {
  pdl_enter();
  using G = Geo<D>;
  constexpr int kA = Alph<W>::kA;
  constexpr int kStage = DecStage<D>::kWords;
  __shared__ __align__(16) uint16_t s_lut[1 << kLutBits];
  __shared__ __align__(16) uint32_t s_words[kStage + 1];
  __shared__ float s_val[kA];
  __shared__ uint32_t s_first[kLmax + 1], s_count[kLmax + 1], s_offset[kLmax + 1];
  __shared__ uint16_t s_sorted[kA];
  __shared__ unsigned long long s_lo, s_hi;
  __shared__ int s_abort;
  Glob* g = w.glob;
  const int tid = threadIdx.x;
  const unsigned int slot = blockIdx.x;   // run slot of this CTA
  // the run, and whether the decode was aborted (then the run map may be
  // stale): one decision for the whole CTA, taken before the run is used
  if (tid == 0) s_abort = dec_aborted(g, epoch);
  const unsigned long long nslots = __ldcg(&g->n_chunks) / kDecRun + (unsigned long long)sh.U;
  uint4 run = make_uint4(~0u, 0u, 0u, 0u);
  if (slot < nslots) run = __ldcg(&w.runmap[slot]);
  __syncthreads();
  if (s_abort || run.x == ~0u) return;
  if (run.x >= (uint32_t)sh.U || run.y >= run.z || run.z > dec_max_chunks(sh)) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_INTERNAL);
    return;
  }
  const int u = (int)run.x;   // unit: slice u / T, table u % T
  const unsigned long long j = (unsigned long long)run.y + tid;
  const bool mine = j < run.z;
  const DecTab* dt = w.dtab + u;
  uint4 dsc = make_uint4(0, 0, 0, 0);
  if (mine) dsc = __ldcg(&w.cdesc[j]);
  {
    const uint4* src = reinterpret_cast<const uint4*>(w.lut + (size_t)u * (1u << kLutBits));
    uint4* dst = reinterpret_cast<uint4*>(s_lut);
#pragma unroll
    for (int i = tid; i < (1 << kLutBits) / 8; i += kDecRun) dst[i] = __ldcg(src + i);
    if (tid <= kLmax) {
      s_first[tid] = __ldcg(&dt->first[tid]);
      s_count[tid] = __ldcg(&dt->count[tid]);
      s_offset[tid] = __ldcg(&dt->offset[tid]);
    }
    const float ebx2 = __ldcg(&dt->ebx2);
#pragma unroll
    for (int i = tid; i < kA; i += kDecRun) {
      s_sorted[i] = dt->sorted[i];
      s_val[i] = __fmul_rn((float)(i - Alph<W>::kR), ebx2);
    }
  }
  // the bitstream of the unit's container
  const unsigned long long n_words = __ldcg(&dt->n_words), off_bits = __ldcg(&dt->bits_off);
  const int t = (int)__ldcg(&dt->t);
  const int64_t slice0 = (int64_t)__ldcg(&dt->row0);
  const uint32_t* words = reinterpret_cast<const uint32_t*>(in + off_bits);
  const unsigned long long start = (unsigned long long)dsc.x | ((unsigned long long)(dsc.y & 0xffffu) << 32);
  const uint32_t clen = dsc.y >> 16;
  const unsigned long long wlim = (start + clen + 31ull) >> 5;   // words the chunk may read: [start/32, wlim)
  if (tid == 0) s_lo = start >> 5;
  if (j + 1 == run.z) s_hi = wlim;
  __syncthreads();
  // the run's words, if they fit (chunk ranges are consecutive by construction;
  // a thread whose range lies outside the staged one reads global memory)
  const unsigned long long lo = s_lo, hi = s_hi;
  const bool staged = hi >= lo && hi - lo <= (unsigned long long)kStage && hi <= n_words;
  if (staged) {
    for (unsigned long long i = lo + tid; i < hi; i += kDecRun) s_words[i - lo] = __ldg(words + i);
    if (tid == 0) s_words[hi - lo] = 0u;   // read past the run's end: a zero word
  }
  __syncthreads();
  if (!mine) return;
  const int seg = (int)dsc.z;
  const uint32_t first = dsc.w & 0xffffu, rows = dsc.w >> 16;
  if (seg / sh.nseg != u || rows == 0u || first + rows > (uint32_t)G::kSB || start + clen > n_words * 32ull) {
    dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  const int s = seg - u * sh.nseg;
  const uint16_t* lrow = w.litrow + (size_t)seg * G::kSB + first;
  const int64_t row0 = slice0 + (int64_t)s * G::kSB;   // batch row of the segment's first row
  bool bad = false;
  unsigned long long used;
  if (staged && (start >> 5) >= lo && wlim <= hi) {
    // reads past the chunk's end see the following chunks' words, then zeros:
    // they never change a code that lies inside the chunk
    const uint32_t* sw = s_words - lo;
    used = decode_chunk<D, W>([&](unsigned long long i) -> uint32_t { return sw[i < hi ? i : hi]; }, start, s_lut,
                           s_val, s_first, s_count, s_offset, s_sorted, lrow, rows, row0, sh.T_out, sh.t_off + t,
                           xhat, &bad);
  } else {
    used = decode_chunk<D, W>([&](unsigned long long i) -> uint32_t { return i < wlim ? __ldg(words + i) : 0u; },
                           start, s_lut, s_val, s_first, s_count, s_offset, s_sorted, lrow, rows, row0, sh.T_out,
                           sh.t_off + t, xhat, &bad);
  }
  if (bad || used != clen) dec_fail(g, epoch, EBC_ERR_CORRUPT);
}

// ---------------------------------------------------------------------------
// k_dec_matches: each matched row copies its reference row: the literal the
// reference names (whole batch), or the literal root of its chain (window;
// resolved by k_dec_prep's table CTAs).  Grid-stride over (matched row,
// 16-byte column) pairs, four copies in flight per thread.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_dec_matches(Shape sh, Work w, float* __restrict__ xhat, uint32_t epoch) {
  pdl_enter();
  Glob* g = w.glob;
  if (dec_aborted(g, epoch)) return;
  constexpr int kQ = D / 4;
  const unsigned long long n4 = __ldcg(&g->n_match) * (unsigned long long)kQ;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  const unsigned long long i_start = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (__ldcg(&g->window) != 0u) {   // source = the chain's literal root
    const uint32_t To = (uint32_t)sh.T_out;   // output rows hold T_out tables; ours start at column t_off
    for (unsigned long long i = i_start; i < n4; i += stride) {
      const uint2 m = __ldcg(&w.mdesc[i / kQ]);
      const unsigned long long q = i % kQ;
      const uint32_t b = m.x / To, col = m.x - b * To;
      const uint32_t from = __ldcg(&w.srcrow[(size_t)(col - (uint32_t)sh.t_off) * sh.B + b]) * To + col;
      __stcs(reinterpret_cast<float4*>(xhat + (size_t)m.x * D + 4 * q),
             *reinterpret_cast<const float4*>(xhat + (size_t)from * D + 4 * q));
    }
    return;
  }
  for (unsigned long long i0 = i_start; i0 < n4; i0 += 4 * stride) {
    float4 v[4];
    unsigned long long dst[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const unsigned long long i = i0 + k * stride;
      if (i < n4) {
        const uint2 m = __ldcg(&w.mdesc[i / kQ]);
        const unsigned long long q = i % kQ;
        v[k] = *reinterpret_cast<const float4*>(xhat + (size_t)m.y * D + 4 * q);
        dst[k] = (size_t)m.x * D + 4 * q;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (i0 + k * stride < n4) __stcs(reinterpret_cast<float4*>(xhat + dst[k]), v[k]);
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D, int W>
static void launch_decompress_d(const uint8_t* in, unsigned long long in_bytes, const unsigned long long* offs,
                                const Shape& sh, const Work& w, float* xhat, uint32_t epoch, cudaStream_t st,
                                Prof* prof) {
  const unsigned nsegT = (unsigned)(sh.U * sh.nseg);
  prof_begin(prof, "k_dec_prep", st);
  launch_k(k_dec_prep<D, W>, (sh.U > 0 ? sh.U : 1) + (nsegT + 7) / 8, 256, 0, st, in, in_bytes, offs, sh, w,
           epoch);
  prof_end(prof, st);
  if (nsegT) {
    // one CTA per run slot: enough for the largest possible chunk count
    prof_begin(prof, "k_dec_chunks", st);
    launch_k(k_dec_chunks<D, W>, (unsigned)(dec_run_slots(sh) - 1), kDecRun, 0, st, in, sh, w, xhat, epoch);
    prof_end(prof, st);
    prof_begin(prof, "k_dec_matches", st);
    static int per_sm = -1;   // resident CTAs per SM: the grid-stride loop runs in one wave
    if (per_sm < 0 &&
        (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dec_matches<D>, 256, 0) != cudaSuccess || per_sm < 1))
      per_sm = 4;
    launch_k(k_dec_matches<D>, (unsigned)((sh.nsm > 0 ? sh.nsm : 152) * per_sm), 256, 0, st, sh, w, xhat, epoch);
    prof_end(prof, st);
  }
}

cudaError_t launch_decompress(const uint8_t* in, unsigned long long in_bytes, const unsigned long long* offs,
                              const Shape& sh, const Work& w, float* xhat, uint32_t epoch, cudaStream_t st,
                              Prof* prof) {
  if (sh.W == 2) {
    switch (sh.D) {
      case 4: launch_decompress_d<4, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 8: launch_decompress_d<8, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 16: launch_decompress_d<16, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 32: launch_decompress_d<32, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 64: launch_decompress_d<64, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 128: launch_decompress_d<128, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 256: launch_decompress_d<256, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      case 512: launch_decompress_d<512, 2>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  switch (sh.D) {
    case 4: launch_decompress_d<4, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 8: launch_decompress_d<8, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 16: launch_decompress_d<16, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 32: launch_decompress_d<32, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 64: launch_decompress_d<64, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 128: launch_decompress_d<128, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 256: launch_decompress_d<256, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    case 512: launch_decompress_d<512, 1>(in, in_bytes, offs, sh, w, xhat, epoch, st, prof); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ebc
