// ebc_decompress.cu -- decompression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (Huffman and vector-based LZ decoding, dequantization) and §III-E
// ("parallel decompression" of chunks).  Three launches:
//   k_dec_tables    validates the header and layout; per table, the canonical
//                   decode tables (2^11-entry first-level table + long codes)
//   k_dec_segments  one CTA per (table, segment); one thread per chunk decodes
//                   into shared memory, then the CTA dequantizes and writes
//                   whole literal rows with 16-byte stores
//   k_dec_matches   copies each matched row from its (literal) reference
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

// ---------------------------------------------------------------------------
// k_dec_tables: grid max(T, 1), 256 threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_dec_tables(const uint8_t* __restrict__ in, unsigned long long in_bytes,
                                                     Shape sh, Work w, uint32_t epoch) {
  __shared__ uint8_t s_len[256];
  __shared__ uint32_t s_count[kLmax + 2], s_next[kLmax + 2], s_offset[kLmax + 2];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int t = blockIdx.x;
  Glob* g = w.glob;
  const int T = sh.T;
  const unsigned long long nvec = (unsigned long long)sh.B * (unsigned long long)T;

  if (t == 0 && tid == 0) {
    int code = EBC_OK;
    if (in_bytes < kHeaderBytes) {
      code = EBC_ERR_CORRUPT;
    } else if (ld32(in) != kMagic || ld32(in + 4) != kFormatVersion) {
      code = EBC_ERR_CORRUPT;
    } else if (ld64(in + 8) != (unsigned long long)sh.B || ld32(in + 16) != (uint32_t)T ||
               ld32(in + 20) != (uint32_t)sh.D) {
      code = EBC_ERR_INVALID_ARG;
    } else if (ld32(in + 24) != (uint32_t)kRadius || ld32(in + 28) != (uint32_t)kLmax ||
               ld32(in + 32) != (uint32_t)sh.SB || ld32(in + 36) != (uint32_t)sh.KC ||
               ld32(in + 40) != (uint32_t)sh.ref_bytes || ld32(in + 44) != 0u) {
      code = EBC_ERR_CORRUPT;
    } else {
      const unsigned long long n_lit = ld64(in + 48), n_match = ld64(in + 56), n_out = ld64(in + 64);
      const unsigned long long n_chunks = ld64(in + 72), words = ld64(in + 80);
      if (n_lit + n_match != nvec || n_lit > nvec || n_chunks > nvec ||
          n_out > nvec * (unsigned long long)sh.D || words > (1ull << 34)) {
        code = EBC_ERR_CORRUPT;
      } else {
        const unsigned long long off_seg = kHeaderBytes + (unsigned long long)T * kTableRecBytes;
        const unsigned long long off_bitmap = off_seg + (unsigned long long)T * sh.nseg * kSegRecBytes;
        const unsigned long long off_chunks = off_bitmap + dpad16((unsigned long long)T * sh.nw * 4ull);
        const unsigned long long off_refs = off_chunks + dpad16(n_chunks * 2ull);
        const unsigned long long off_out = off_refs + dpad16(n_match * (unsigned long long)sh.ref_bytes);
        const unsigned long long off_bits = off_out + dpad16(n_out * 4ull);
        const unsigned long long total = off_bits + words * 4ull;
        if (ld64(in + 88) != off_seg || ld64(in + 96) != off_bitmap || ld64(in + 104) != off_chunks ||
            ld64(in + 112) != off_refs || ld64(in + 120) != off_out || ld64(in + 128) != off_bits ||
            ld64(in + 136) != total || total > in_bytes) {
          code = EBC_ERR_CORRUPT;
        } else {
          g->n_lit = n_lit; g->n_match = n_match; g->n_out = n_out; g->n_chunks = n_chunks; g->words = words;
          g->off_seg = off_seg; g->off_bitmap = off_bitmap; g->off_chunks = off_chunks; g->off_refs = off_refs;
          g->off_out = off_out; g->off_bits = off_bits; g->total = total;
        }
      }
    }
    if (code != EBC_OK) dec_fail(g, epoch, code);
  }
  if (t >= T) return;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (kHeaderBytes + (unsigned long long)T * kTableRecBytes > in_bytes) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  const uint8_t* rec = in + kHeaderBytes + (size_t)t * kTableRecBytes;
  const uint32_t L = rec[16 + tid];
  s_len[tid] = (uint8_t)L;
  if (tid < kLmax + 2) s_count[tid] = 0;
  __syncthreads();
  if (L > (uint32_t)kLmax) s_bad = 1;
  else if (L) atomicAdd(&s_count[L], 1u);
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
  if (L) {
    uint32_t rank = 0;
    for (int j = 0; j < tid; ++j) rank += (s_len[j] == L);
    const uint32_t code = s_next[L] + rank;
    w.dtab[t].sorted[s_offset[L] + rank] = (uint8_t)tid;
    if (L <= (uint32_t)kLutBits) {
      const uint32_t lo = code << (kLutBits - L), n = 1u << (kLutBits - L);
      for (uint32_t i = 0; i < n; ++i) lut[lo + i] = (uint16_t)(tid | (L << 8));
    }
  }
}

// ---------------------------------------------------------------------------
// k_dec_segments: one CTA (64 threads) per (table, segment).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(64) k_dec_segments(const uint8_t* __restrict__ in, Shape sh, Work w,
                                                      float* __restrict__ xhat, uint32_t epoch) {
  using G = Geo<D>;
  constexpr int kThreads = 64;
  __shared__ __align__(16) uint16_t s_lut[1 << kLutBits];
  __shared__ __align__(16) uint16_t s_stage[G::kSegSyms];
  __shared__ uint16_t s_litrow[G::kSB];
  __shared__ float s_deq[256];
  __shared__ uint32_t s_first[kLmax + 1], s_count[kLmax + 1], s_offset[kLmax + 1];
  __shared__ uint8_t s_sorted[256];
  __shared__ uint32_t s_cstart[G::kChunks + 1];
  __shared__ uint32_t s_cout[G::kChunks + 1];
  __shared__ uint32_t s_wpre[kThreads];
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
  const unsigned long long off_chunks = __ldcg(&g->off_chunks), off_out = __ldcg(&g->off_out);
  const unsigned long long off_bits = __ldcg(&g->off_bits);
  const unsigned long long n_chunks = __ldcg(&g->n_chunks), n_out = __ldcg(&g->n_out);
  const unsigned long long n_words = __ldcg(&g->words);
  const uint32_t* rec = reinterpret_cast<const uint32_t*>(in + off_seg + (unsigned long long)seg * kSegRecBytes);
  const uint32_t word_off = rec[0], chunk_base = rec[1], out_base = rec[3];

  {  // decode tables of this table
    const uint4* src = reinterpret_cast<const uint4*>(w.lut + (size_t)t * (1u << kLutBits));
    uint4* dst = reinterpret_cast<uint4*>(s_lut);
    for (int i = tid; i < (1 << kLutBits) / 8; i += kThreads) dst[i] = __ldcg(src + i);
    const DecTab* dt = w.dtab + t;
    if (tid <= kLmax) {
      s_first[tid] = dt->first[tid];
      s_count[tid] = dt->count[tid];
      s_offset[tid] = dt->offset[tid];
    }
    const float ebx2 = dt->ebx2;
    for (int i = tid; i < 256; i += kThreads) {
      s_sorted[i] = dt->sorted[i];
      s_deq[i] = __fmul_rn((float)(i - kRadius), ebx2);
    }
  }
  if (tid == 0) s_bad = 0;
  // literal rows of the segment, in row order
  uint32_t litw = 0;
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    if (wi < sh.nw) {
      const uint32_t bm = ld32(in + off_bitmap + 4ull * ((size_t)t * sh.nw + wi));
      const int64_t first_row = row0 + tid * 32;
      const int64_t nvalid = B - first_row;
      const uint32_t vmask = nvalid >= 32 ? 0xffffffffu : ((1u << nvalid) - 1u);
      litw = ~bm & vmask;
    }
  }
  s_wpre[tid] = __popc(litw);
  __syncthreads();
  if (tid == 0) {
    uint32_t acc = 0;
    for (int i = 0; i < kThreads; ++i) {
      const uint32_t c = s_wpre[i];
      s_wpre[i] = acc;
      acc += c;
    }
    s_cstart[G::kChunks] = acc;  // temporarily: literal count
  }
  __syncthreads();
  const uint32_t nlit = s_cstart[G::kChunks];
  {
    uint32_t k = s_wpre[tid], m = litw;
    while (m) {
      const int bit = __ffs(m) - 1;
      s_litrow[k++] = (uint16_t)(tid * 32 + bit);
      m &= m - 1;
    }
  }
  const uint32_t nchunks = (nlit + G::kKC - 1) / G::kKC;
  __syncthreads();
  if ((unsigned long long)chunk_base + nchunks > n_chunks) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  // chunk start bits (relative to the segment)
  if (tid == 0) {
    uint32_t acc = 0;
    const uint16_t* cl = reinterpret_cast<const uint16_t*>(in + off_chunks) + chunk_base;
    for (uint32_t c = 0; c < nchunks; ++c) {
      s_cstart[c] = acc;
      acc += cl[c];
    }
    s_cstart[nchunks] = acc;
    const unsigned long long seg_words = ((acc + 127ull) >> 7) * 4ull;
    if ((unsigned long long)word_off + seg_words > n_words) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  const uint32_t seg_bits = s_cstart[nchunks];
  const unsigned long long wlim = (unsigned long long)word_off + ((seg_bits + 127ull) >> 7) * 4ull;

  // decode: thread c decodes chunk c
  if ((uint32_t)tid < nchunks) {
    const uint32_t c = tid;
    const uint32_t rows = min((uint32_t)G::kKC, nlit - c * G::kKC);
    const uint32_t nsym = rows * D;
    const uint32_t* words = reinterpret_cast<const uint32_t*>(in + off_bits);
    const unsigned long long start = (unsigned long long)word_off * 32ull + s_cstart[c];
    const uint32_t clen = s_cstart[c + 1] - s_cstart[c];
    unsigned long long wp = start >> 5;
    auto ldw = [&](unsigned long long i) -> unsigned long long {
      return i < wlim ? (unsigned long long)__ldg(words + i) : 0ull;
    };
    unsigned long long buf = (ldw(wp) << 32) | ldw(wp + 1);
    const uint32_t skip = (uint32_t)(start & 31ull);
    buf <<= skip;
    int nb = 64 - (int)skip;
    wp += 2;
    uint32_t used = 0, nout = 0;
    bool bad = false;
    uint16_t* dst = s_stage + c * G::kKC * D;
    for (uint32_t i = 0; i < nsym; ++i) {
      if (nb < 32) {
        buf |= ldw(wp++) << (32 - nb);
        nb += 32;
      }
      const uint32_t e = s_lut[buf >> (64 - kLutBits)];
      uint32_t len = e >> 8, sym = e & 0xffu;
      if (len == 0u) {
        for (int l = kLutBits + 1; l <= kLmax; ++l) {
          const uint32_t code = (uint32_t)(buf >> (64 - l));
          if (code - s_first[l] < s_count[l]) {
            sym = s_sorted[s_offset[l] + code - s_first[l]];
            len = (uint32_t)l;
            break;
          }
        }
        if (len == 0u) { bad = true; break; }
      }
      buf <<= len;
      nb -= (int)len;
      used += len;
      dst[i] = sym ? (uint16_t)sym : (uint16_t)(0x8000u | nout++);
    }
    if (bad || used != clen) s_bad = 1;
    s_cout[c] = nout;
  }
  __syncthreads();
  if (tid == 0 && !s_bad) {
    uint32_t acc = 0;
    for (uint32_t c = 0; c < nchunks; ++c) {
      const uint32_t v = s_cout[c];
      s_cout[c] = acc;
      acc += v;
    }
    if ((unsigned long long)out_base + acc > n_out) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  // dequantize and write whole literal rows
  const uint32_t* outl = reinterpret_cast<const uint32_t*>(in + off_out) + out_base;
  const uint32_t n4 = nlit * (D / 4);
  for (uint32_t i = tid; i < n4; i += kThreads) {
    const uint32_t li = i / (D / 4);
    const uint32_t d = (i % (D / 4)) * 4;
    const int64_t b = row0 + s_litrow[li];
    const uint2 pk = *reinterpret_cast<const uint2*>(s_stage + li * D + d);
    const uint32_t v0 = pk.x & 0xffffu, v1 = pk.x >> 16, v2 = pk.y & 0xffffu, v3 = pk.y >> 16;
    const uint32_t ob = s_cout[li / G::kKC];
    float4 o;
    o.x = v0 & 0x8000u ? __uint_as_float(__ldg(outl + ob + (v0 & 0x7fffu))) : s_deq[v0];
    o.y = v1 & 0x8000u ? __uint_as_float(__ldg(outl + ob + (v1 & 0x7fffu))) : s_deq[v1];
    o.z = v2 & 0x8000u ? __uint_as_float(__ldg(outl + ob + (v2 & 0x7fffu))) : s_deq[v2];
    o.w = v3 & 0x8000u ? __uint_as_float(__ldg(outl + ob + (v3 & 0x7fffu))) : s_deq[v3];
    __stcs(reinterpret_cast<float4*>(xhat + ((size_t)b * T + t) * D + d), o);
  }
}

// ---------------------------------------------------------------------------
// k_dec_matches: one CTA per (table, segment); each matched row copies its
// reference row, which is always a literal of the same table and earlier.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_dec_matches(const uint8_t* __restrict__ in, Shape sh, Work w,
                                                      float* __restrict__ xhat, uint32_t epoch) {
  using G = Geo<D>;
  __shared__ uint32_t s_bm[G::kBmWords];
  __shared__ uint32_t s_pre[G::kBmWords + 1];
  __shared__ int s_bad;
  Glob* g = w.glob;
  if (dec_aborted(g, epoch)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  if (tid == 0) {
    uint32_t acc = 0;
    for (int i = 0; i < G::kBmWords; ++i) {
      s_pre[i] = acc;
      acc += __popc(s_bm[i]);
    }
    s_pre[G::kBmWords] = acc;
    if ((unsigned long long)match_base + acc > n_match) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
    return;
  }
  const uint8_t* refs = in + off_refs;
#pragma unroll 1
  for (int it = 0; it < G::kRowsPerWarp / G::kRPS; ++it) {
    const int r = warp * G::kRowsPerWarp + it * G::kRPS + lane / G::kLPR;
    const int64_t b = row0 + r;
    const bool m = b < B && ((s_bm[r >> 5] >> (r & 31)) & 1u);
    if (!m) continue;
    const uint32_t rank = s_pre[r >> 5] + __popc(s_bm[r >> 5] & ((1u << (r & 31)) - 1u));
    const unsigned long long mi = (unsigned long long)match_base + rank;
    const uint32_t ref = sh.ref_bytes == 2 ? (uint32_t)reinterpret_cast<const uint16_t*>(refs)[mi]
                                           : reinterpret_cast<const uint32_t*>(refs)[mi];
    if ((int64_t)ref >= b || ((bmt[ref >> 5] >> (ref & 31)) & 1u)) {
      dec_fail(g, epoch, EBC_ERR_CORRUPT);
      continue;
    }
    const float* src = xhat + ((size_t)ref * T + t) * D;
    float* dst = xhat + ((size_t)b * T + t) * D;
#pragma unroll
    for (int j = 0; j < G::kSPR; ++j) {
      const int d = (lane % G::kLPR) * 4 + j * 128;
      __stcs(reinterpret_cast<float4*>(dst + d), *reinterpret_cast<const float4*>(src + d));
    }
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D>
static void launch_decompress_d(const uint8_t* in, unsigned long long in_bytes, const Shape& sh, const Work& w,
                                float* xhat, uint32_t epoch, cudaStream_t st, Prof* prof) {
  prof_begin(prof, "k_dec_tables", st);
  k_dec_tables<<<sh.T > 0 ? sh.T : 1, 256, 0, st>>>(in, in_bytes, sh, w, epoch);
  prof_end(prof, st);
  const unsigned grid = (unsigned)(sh.T * sh.nseg);
  if (grid) {
    prof_begin(prof, "k_dec_segments", st);
    k_dec_segments<D><<<grid, 64, 0, st>>>(in, sh, w, xhat, epoch);
    prof_end(prof, st);
    prof_begin(prof, "k_dec_matches", st);
    k_dec_matches<D><<<grid, 256, 0, st>>>(in, sh, w, xhat, epoch);
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
