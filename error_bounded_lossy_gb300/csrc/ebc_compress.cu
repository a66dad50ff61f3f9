// ebc_compress.cu -- compression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (quantization encoder, vector-based LZ, Huffman) and §III-E (one
// output buffer).  Four launches on the caller's stream, each over the
// (table, segment) grid except the codebook kernel:
//   k_quantize  x -> codes, per-vector dedup key, first-occurrence hash table
//   k_resolve   literal / match decision, per-segment literal histogram, bitmap
//   k_codebook  per-table Huffman code + segment offsets; the last CTA lays out
//               the container (header, section offsets, size)
//   k_emit      bitstream, chunk index, references, outliers, segment records
// All offsets come from prefix sums, never from atomics, so the container is
// byte-identical from run to run.
#include <cstdint>

#include "ebc_internal.cuh"

namespace ebc {

// ---------------------------------------------------------------------------
// Quantization encoder (§III-D), no predictor (§III-B observation 1): the code
// is q + 128 with q = round_half_even(x * fl32(1 / 2eb)), accepted when
// |q| < 128 and |x - fl32(q * 2eb)| <= eb in fp32; otherwise 0 (outlier).
// Rounding to the nearest integer adds 1.5 * 2^23, which leaves the integer in
// the low mantissa bits (valid for |t| < 2^22; larger |t| were rejected).
// Every operation is an explicitly rounded intrinsic, so nothing is contracted.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quantize_one(float x, float eb, float ebx2, float inv) {
  const float t = __fmul_rn(x, inv);
  if (!(fabsf(t) < 127.5f)) return 0u;             // NaN, +-inf, |q| >= 128
  const float y = __fadd_rn(t, 12582912.0f);       // 1.5 * 2^23
  const float qf = __fsub_rn(y, 12582912.0f);      // exact
  const float xh = __fmul_rn(qf, ebx2);
  const float err = fabsf(__fsub_rn(x, xh));
  if (!(err <= eb)) return 0u;
  return (uint32_t)(__float_as_int(y) - 0x4B400000 + kRadius);
}

__device__ __forceinline__ void dedup_insert(unsigned long long* slots, uint32_t S, uint32_t h,
                                             uint32_t b, Glob* g) {
  // First occurrence per key: the slot keeps (h << 32 | min row); keys that
  // collide on the slot index probe linearly.
  const unsigned long long mine = ((unsigned long long)h << 32) | b;
  uint32_t slot = h & (S - 1);
  for (uint32_t p = 0; p < S; ++p) {
    const unsigned long long old = atomicCAS(slots + slot, kEmptySlot, mine);
    if (old == kEmptySlot) return;
    if ((uint32_t)(old >> 32) == h) {
      if (old > mine) atomicMin(slots + slot, mine);
      return;
    }
    slot = (slot + 1) & (S - 1);
  }
  record_error(g, EBC_ERR_INTERNAL);
}

__device__ __forceinline__ uint32_t dedup_lookup(const unsigned long long* slots, uint32_t S,
                                                 uint32_t h, Glob* g) {
  uint32_t slot = h & (S - 1);
  for (uint32_t p = 0; p < S; ++p) {
    const unsigned long long v = slots[slot];
    if (v == kEmptySlot) break;
    if ((uint32_t)(v >> 32) == h) return (uint32_t)v;
    slot = (slot + 1) & (S - 1);
  }
  record_error(g, EBC_ERR_INTERNAL);
  return 0xFFFFFFFFu;
}

// ---------------------------------------------------------------------------
// k_quantize: one CTA per (table, segment), 8 warps, each warp a run of
// 128-element slabs (lane = 4 consecutive elements, one 16-byte load).
// The dedup key of a vector is the wrapping sum over its 4-code words w_k of
// lowbias32(w_k + k * 0x9E3779B9) plus lowbias32(raw ^ (d + 1) * 0x85EBCA6B)
// for each outlier at position d.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_quantize(const float* __restrict__ x, Shape sh, EbParams ep,
                                                   Work w) {
  using G = Geo<D>;
  const int seg = blockIdx.x;
  const int t = seg / sh.nseg;
  const int s = seg - t * sh.nseg;
  const float eb = ep.eb[t];
  const float ebx2 = __fmul_rn(2.0f, eb);
  const float inv = __fdiv_rn(1.0f, ebx2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t B = sh.B;
  const int T = sh.T;
  const int64_t row0 = (int64_t)s * G::kSB;
  unsigned long long* slots = w.slots + (size_t)t * sh.S;
  uint32_t acc = 0, nout = 0;
  constexpr int kBatch = 8;
#pragma unroll 1
  for (int i0 = 0; i0 < G::kSlabsPerWarp; i0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int e = (warp * G::kSlabsPerWarp + i0 + k) * 128 + lane * 4;
      const int64_t b = row0 + e / D;
      const int d = e % D;
      v[k] = b < B ? ld_stream_f4(x + ((size_t)(b * T + t) * D + d)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int slab = warp * G::kSlabsPerWarp + i0 + k;
      const int e = slab * 128 + lane * 4;
      const int64_t b = row0 + e / D;
      const int d = e % D;
      const bool valid = b < B;
      const uint32_t c0 = quantize_one(v[k].x, eb, ebx2, inv);
      const uint32_t c1 = quantize_one(v[k].y, eb, ebx2, inv);
      const uint32_t c2 = quantize_one(v[k].z, eb, ebx2, inv);
      const uint32_t c3 = quantize_one(v[k].w, eb, ebx2, inv);
      const uint32_t word = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
      if (valid) *reinterpret_cast<uint32_t*>(w.sym + ((size_t)t * B + b) * D + d) = word;
      acc += lowbias32(word + (uint32_t)(d >> 2) * 0x9E3779B9u);
      if ((c0 == 0u) | (c1 == 0u) | (c2 == 0u) | (c3 == 0u)) {
        if (c0 == 0u) { acc += lowbias32(__float_as_uint(v[k].x) ^ (uint32_t)(d + 1) * 0x85EBCA6Bu); ++nout; }
        if (c1 == 0u) { acc += lowbias32(__float_as_uint(v[k].y) ^ (uint32_t)(d + 2) * 0x85EBCA6Bu); ++nout; }
        if (c2 == 0u) { acc += lowbias32(__float_as_uint(v[k].z) ^ (uint32_t)(d + 3) * 0x85EBCA6Bu); ++nout; }
        if (c3 == 0u) { acc += lowbias32(__float_as_uint(v[k].w) ^ (uint32_t)(d + 4) * 0x85EBCA6Bu); ++nout; }
      }
      if ((slab + 1) % G::kSPR == 0) {            // the row ends with this slab
#pragma unroll
        for (int off = G::kLPR / 2; off > 0; off >>= 1) {
          acc += __shfl_xor_sync(0xffffffffu, acc, off);
          nout += __shfl_xor_sync(0xffffffffu, nout, off);
        }
        if (valid && (lane % G::kLPR) == 0) {
          w.vhash[(size_t)t * B + b] = acc;
          w.vnout[(size_t)t * B + b] = nout;
          dedup_insert(slots, sh.S, acc, (uint32_t)b, w.glob);
        }
        acc = 0;
        nout = 0;
      }
    }
  }
}

__device__ __forceinline__ bool has_zero_byte(uint32_t v) {
  return ((v - 0x01010101u) & ~v & 0x80808080u) != 0u;
}

// ---------------------------------------------------------------------------
// k_resolve: vector-based LZ with the whole batch as window and the first
// occurrence as reference (§III-D, §III-E "fixed pattern length"): row b is a
// match when the first row with its key precedes it and carries the same codes
// and the same raw bits at outliers; otherwise a literal (a key collision is
// a literal too).  Literal codes feed the segment histogram.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_resolve(const float* __restrict__ x, Shape sh, Work w) {
  using G = Geo<D>;
  __shared__ uint32_t s_hist[8][256];
  __shared__ uint32_t s_bm[G::kBmWords];
  __shared__ uint32_t s_cnt[3];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 8 * 256; i += 256) (&s_hist[0][0])[i] = 0u;
  if (tid < G::kBmWords) s_bm[tid] = 0u;
  if (tid < 3) s_cnt[tid] = 0u;
  __syncthreads();

  const int seg = blockIdx.x;
  const int t = seg / sh.nseg;
  const int s = seg - t * sh.nseg;
  const int64_t B = sh.B;
  const int T = sh.T;
  const int64_t row0 = (int64_t)s * G::kSB;
  const unsigned long long* slots = w.slots + (size_t)t * sh.S;
  const uint8_t* symt = w.sym + (size_t)t * B * D;
  uint32_t* hist = s_hist[warp];
  const unsigned gshift = lane & ~(G::kLPR - 1);
  const unsigned gmask = (G::kLPR == 32 ? 0xffffffffu : ((1u << G::kLPR) - 1u)) << gshift;
  const bool leader = (lane % G::kLPR) == 0;
  uint32_t n_lit = 0, n_match = 0, n_out = 0;

#pragma unroll 1
  for (int it = 0; it < G::kRowsPerWarp / G::kRPS; ++it) {
    const int r = warp * G::kRowsPerWarp + it * G::kRPS + lane / G::kLPR;
    const int64_t b = row0 + r;
    const bool valid = b < B;
    uint32_t ref = (uint32_t)b;
    if (valid && leader) {
      ref = dedup_lookup(slots, sh.S, w.vhash[(size_t)t * B + b], w.glob);
      if (ref > (uint32_t)b) ref = (uint32_t)b;   // only on an internal error
    }
    ref = __shfl_sync(0xffffffffu, ref, gshift);
    uint32_t wb[G::kSPR];
    bool eq = true;
#pragma unroll
    for (int j = 0; j < G::kSPR; ++j) {
      const int d = (lane % G::kLPR) * 4 + j * 128;
      wb[j] = valid ? *reinterpret_cast<const uint32_t*>(symt + (size_t)b * D + d) : 0u;
      if (valid && ref != (uint32_t)b) {
        const uint32_t wr = *reinterpret_cast<const uint32_t*>(symt + (size_t)ref * D + d);
        bool e = wr == wb[j];
        if (e && has_zero_byte(wb[j])) {
          const float* xb = x + ((size_t)b * T + t) * D + d;
          const float* xr = x + ((size_t)ref * T + t) * D + d;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (((wb[j] >> (8 * q)) & 0xffu) == 0u && __float_as_uint(xb[q]) != __float_as_uint(xr[q])) e = false;
        }
        eq = eq && e;
      }
    }
    const unsigned bad = __ballot_sync(0xffffffffu, !eq);
    const bool match = valid && ref != (uint32_t)b && (bad & gmask) == 0u;
    if (valid && !match) {
#pragma unroll
      for (int j = 0; j < G::kSPR; ++j) {
        atomicAdd(&hist[wb[j] & 0xffu], 1u);
        atomicAdd(&hist[(wb[j] >> 8) & 0xffu], 1u);
        atomicAdd(&hist[(wb[j] >> 16) & 0xffu], 1u);
        atomicAdd(&hist[wb[j] >> 24], 1u);
      }
    }
    if (valid && leader) {
      w.ref[(size_t)t * B + b] = match ? ref : (uint32_t)b;
      if (match) {
        atomicOr(&s_bm[r >> 5], 1u << (r & 31));
        ++n_match;
      } else {
        ++n_lit;
        n_out += w.vnout[(size_t)t * B + b];
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    n_lit += __shfl_xor_sync(0xffffffffu, n_lit, off);
    n_match += __shfl_xor_sync(0xffffffffu, n_match, off);
    n_out += __shfl_xor_sync(0xffffffffu, n_out, off);
  }
  if (lane == 0) {
    atomicAdd(&s_cnt[0], n_lit);
    atomicAdd(&s_cnt[1], n_match);
    atomicAdd(&s_cnt[2], n_out);
  }
  __syncthreads();
  uint32_t f = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) f += s_hist[k][tid];
  w.seg_hist[(size_t)seg * 256 + tid] = f;
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    if (wi < sh.nw) w.bitmap[(size_t)t * sh.nw + wi] = s_bm[tid];
  }
  if (tid == 0)
    w.seg_cnt[seg] = make_uint4(s_cnt[0], s_cnt[1], s_cnt[2], (s_cnt[0] + G::kKC - 1) / G::kKC);
}

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of uint4 over 256 threads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 add4(uint4 a, uint4 b) {
  return make_uint4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ uint4 block_excl_scan4(uint4 v, uint4* total, uint4* s_warp) {
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

__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ void st_u64(uint8_t* p, unsigned long long v) {
  *reinterpret_cast<unsigned long long*>(p) = v;
}
__device__ __forceinline__ unsigned long long pad16(unsigned long long n) { return (n + 15ull) & ~15ull; }

// ---------------------------------------------------------------------------
// k_codebook: one CTA per table.  Huffman code lengths (§III-D "Optimized
// Entropy Encoding") by the two-queue construction over leaves sorted by
// (count, symbol), merged nodes in FIFO order, ties to the leaf; if the longest
// code exceeds 24 bits every nonzero count becomes max(1, count >> 1) and the
// code is rebuilt.  Canonical code values follow the DEFLATE rule.  Then the
// per-segment bit counts come from the segment histograms and one exclusive
// scan gives each segment's table-relative offsets.  The last CTA to finish
// sums the tables and writes the header.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_codebook(Shape sh, EbParams ep, Work w, uint8_t* __restrict__ out,
                                                   unsigned long long cap, unsigned long long* out_bytes,
                                                   uint32_t epoch) {
  __shared__ uint32_t s_f[256];
  __shared__ uint16_t s_order[256];
  __shared__ uint32_t s_nodew[256];
  __shared__ uint8_t s_leafpar[256], s_nodepar[256], s_depth[256], s_len[256];
  __shared__ uint32_t s_count[kLmax + 2], s_next[kLmax + 2];
  __shared__ int s_maxlen;
  __shared__ uint32_t s_bits[256];
  __shared__ uint4 s_warp[8];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int T = sh.T;

  if (t < T) {
    const size_t seg0 = (size_t)t * sh.nseg;
    uint32_t f = 0;
    for (int g = 0; g < sh.nseg; ++g) f += __ldcg(&w.seg_hist[(seg0 + g) * 256 + tid]);
    s_f[tid] = f;
    __syncthreads();
    for (int round = 0; round < 40; ++round) {
      const uint32_t fi = s_f[tid];
      int rank = 0;
      if (fi > 0u)
        for (int j = 0; j < 256; ++j) {
          const uint32_t fj = s_f[j];
          rank += (fj > 0u) && (fj < fi || (fj == fi && j < tid));
        }
      const int n = __syncthreads_count(fi > 0u);
      if (fi > 0u) s_order[rank] = (uint16_t)tid;
      s_len[tid] = 0;
      __syncthreads();
      if (tid == 0) {
        int maxlen = 0;
        if (n == 1) {
          s_len[s_order[0]] = 1;
          maxlen = 1;
        } else if (n >= 2) {
          int li = 0, qi = 0, qn = 0;
          for (int m = 0; m < n - 1; ++m) {
            uint32_t wsum = 0;
            for (int pick = 0; pick < 2; ++pick) {
              const bool leaf = li < n && (qi >= qn || s_f[s_order[li]] <= s_nodew[qi]);
              if (leaf) {
                s_leafpar[li] = (uint8_t)m;
                wsum += s_f[s_order[li]];
                ++li;
              } else {
                s_nodepar[qi] = (uint8_t)m;
                wsum += s_nodew[qi];
                ++qi;
              }
            }
            s_nodew[qn++] = wsum;
          }
          s_depth[n - 2] = 0;
          for (int m = n - 3; m >= 0; --m) s_depth[m] = (uint8_t)(s_depth[s_nodepar[m]] + 1);
          for (int i = 0; i < n; ++i) {
            const int l = s_depth[s_leafpar[i]] + 1;
            s_len[s_order[i]] = (uint8_t)l;
            maxlen = l > maxlen ? l : maxlen;
          }
        }
        s_maxlen = maxlen;
      }
      __syncthreads();
      if (s_maxlen <= kLmax) break;
      if (fi > 0u) s_f[tid] = (fi >> 1) > 0u ? (fi >> 1) : 1u;
      __syncthreads();
    }
    // canonical codes
    if (tid < kLmax + 2) s_count[tid] = 0;
    __syncthreads();
    const uint32_t L = s_len[tid];
    if (L) atomicAdd(&s_count[L], 1u);
    __syncthreads();
    if (tid == 0) {
      uint32_t c = 0;
      s_count[0] = 0;
      for (int l = 1; l <= kLmax; ++l) {
        c = (c + s_count[l - 1]) << 1;
        s_next[l] = c;
      }
    }
    __syncthreads();
    uint32_t code = 0;
    if (L) {
      code = s_next[L];
      for (int j = 0; j < tid; ++j) code += (s_len[j] == L);
    }
    w.tabcode[(size_t)t * 256 + tid] = (code << 8) | L;
    uint8_t* rec = out + kHeaderBytes + (size_t)t * kTableRecBytes;
    rec[16 + tid] = (uint8_t)L;

    // per-segment bits and offsets
    uint4 carry = make_uint4(0, 0, 0, 0);
    uint32_t lits = 0;
    for (int base = 0; base < sh.nseg; base += 256) {
      for (int k = warp; k < 256; k += 8) {
        const int g = base + k;
        uint32_t bsum = 0;
        if (g < sh.nseg) {
          const uint32_t* h = w.seg_hist + (seg0 + g) * 256;
          for (int j = lane; j < 256; j += 32) bsum += __ldcg(h + j) * (uint32_t)s_len[j];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, off);
        if (lane == 0) s_bits[k] = bsum;
      }
      __syncthreads();
      const int g = base + tid;
      uint4 v = make_uint4(0, 0, 0, 0);
      uint32_t nl = 0;
      if (g < sh.nseg) {
        const uint4 c = __ldcg(&w.seg_cnt[seg0 + g]);
        const uint32_t words = ((s_bits[tid] + 127u) >> 7) * 4u;
        v = make_uint4(words, c.w, c.y, c.z);
        nl = c.x;
        w.seg_words[seg0 + g] = words;
      }
      uint4 tot;
      const uint4 ex = block_excl_scan4(make_uint4(v.x, v.y, v.z, v.w), &tot, s_warp);
      if (g < sh.nseg) w.seg_off[seg0 + g] = add4(carry, ex);
      carry = add4(carry, tot);
      uint4 ltot;
      block_excl_scan4(make_uint4(nl, 0, 0, 0), &ltot, s_warp);
      lits += ltot.x;
    }
    if (tid == 0) {
      w.tab_tot[t] = carry;
      w.tab_lits[t] = lits;
      st_u32(rec + 0, __float_as_uint(ep.eb[t]));
      st_u32(rec + 4, lits);
      st_u32(rec + 8, carry.z);
      st_u32(rec + 12, carry.w);
    }
  }

  // ---- the last CTA: table bases, layout and header ----
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&w.glob->done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint4 carry = make_uint4(0, 0, 0, 0);
  unsigned long long lits = 0;
  for (int base = 0; base < T; base += 256) {
    const int i = base + tid;
    const uint4 v = i < T ? __ldcg(&w.tab_tot[i]) : make_uint4(0, 0, 0, 0);
    const uint32_t nl = i < T ? __ldcg(&w.tab_lits[i]) : 0u;
    uint4 tot;
    const uint4 ex = block_excl_scan4(v, &tot, s_warp);
    if (i < T) w.tab_base[i] = add4(carry, ex);
    carry = add4(carry, tot);
    uint4 ltot;
    block_excl_scan4(make_uint4(nl, 0, 0, 0), &ltot, s_warp);
    lits += ltot.x;
  }
  if (tid == 0) {
    Glob* g = w.glob;
    const unsigned long long words = carry.x, chunks = carry.y, matches = carry.z, outl = carry.w;
    const unsigned long long off_seg = kHeaderBytes + (unsigned long long)T * kTableRecBytes;
    const unsigned long long off_bitmap = off_seg + (unsigned long long)T * sh.nseg * kSegRecBytes;
    const unsigned long long bm_bytes = (unsigned long long)T * sh.nw * 4ull;
    const unsigned long long off_chunks = off_bitmap + pad16(bm_bytes);
    const unsigned long long off_refs = off_chunks + pad16(chunks * 2ull);
    const unsigned long long off_out = off_refs + pad16(matches * (unsigned long long)sh.ref_bytes);
    const unsigned long long off_bits = off_out + pad16(outl * 4ull);
    const unsigned long long total = off_bits + words * 4ull;
    g->n_lit = lits; g->n_match = matches; g->n_out = outl; g->n_chunks = chunks; g->words = words;
    g->off_seg = off_seg; g->off_bitmap = off_bitmap; g->off_chunks = off_chunks; g->off_refs = off_refs;
    g->off_out = off_out; g->off_bits = off_bits; g->total = total;
    *out_bytes = total;
    const int status = total > cap ? EBC_ERR_CAPACITY : EBC_OK;
    st_u32(out + 0, kMagic); st_u32(out + 4, kFormatVersion); st_u64(out + 8, (unsigned long long)sh.B);
    st_u32(out + 16, (uint32_t)T); st_u32(out + 20, (uint32_t)sh.D); st_u32(out + 24, kRadius);
    st_u32(out + 28, kLmax); st_u32(out + 32, (uint32_t)sh.SB); st_u32(out + 36, (uint32_t)sh.KC);
    st_u32(out + 40, (uint32_t)sh.ref_bytes); st_u32(out + 44, 0u);
    st_u64(out + 48, lits); st_u64(out + 56, matches); st_u64(out + 64, outl); st_u64(out + 72, chunks);
    st_u64(out + 80, words); st_u64(out + 88, off_seg); st_u64(out + 96, off_bitmap);
    st_u64(out + 104, off_chunks); st_u64(out + 112, off_refs); st_u64(out + 120, off_out);
    st_u64(out + 128, off_bits); st_u64(out + 136, total);
    if (status == EBC_OK) {
      // zero the alignment padding after each variable-length section
      for (unsigned long long i = off_bitmap + bm_bytes; i < off_chunks; ++i) out[i] = 0;
      for (unsigned long long i = off_chunks + chunks * 2ull; i < off_refs; ++i) out[i] = 0;
      for (unsigned long long i = off_refs + matches * sh.ref_bytes; i < off_out; ++i) out[i] = 0;
      for (unsigned long long i = off_out + outl * 4ull; i < off_bits; ++i) out[i] = 0;
    } else {
      record_error(g, status);
    }
    g->cstat = status_word(epoch, status);
    g->done = 0u;
  }
}

// Writes `len` bits of `code` MSB-first at bit position p of a word array.
__device__ __forceinline__ void put_bits(uint32_t* s, uint32_t p, uint32_t code, uint32_t len) {
  const uint32_t sh = p & 31u;
  const unsigned long long v = (unsigned long long)code << (64u - len - sh);
  atomicOr(&s[p >> 5], (uint32_t)(v >> 32));
  const uint32_t lo = (uint32_t)v;
  if (lo) atomicOr(&s[(p >> 5) + 1], lo);
}

// ---------------------------------------------------------------------------
// k_emit: one CTA per (table, segment).  Codes are written MSB-first into a
// shared-memory copy of the segment's bitstream (offsets from a prefix sum of
// the per-row bit counts), then stored with 16-byte writes.  Also writes the
// segment's chunk lengths, references, outliers, record and bitmap words.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_emit(const float* __restrict__ x, Shape sh, Work w,
                                               uint8_t* __restrict__ out, uint32_t epoch) {
  using G = Geo<D>;
  extern __shared__ __align__(16) uint32_t s_bits[];
  __shared__ uint32_t s_code[256];
  __shared__ uint32_t s_bm[G::kBmWords];
  __shared__ uint32_t s_rowoff[G::kSB];
  __shared__ uint32_t s_aux[G::kSB];
  __shared__ uint16_t s_litrow[G::kSB];
  __shared__ uint4 s_warp[8];
  __shared__ uint32_t s_segbits;
  if (__ldcg(&w.glob->cstat) != status_word(epoch, EBC_OK)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x;
  const int t = seg / sh.nseg;
  const int s = seg - t * sh.nseg;
  const int64_t B = sh.B;
  const int T = sh.T;
  const int64_t row0 = (int64_t)s * G::kSB;
  const uint8_t* symt = w.sym + (size_t)t * B * D;
  const uint4 base = add4(__ldcg(&w.tab_base[t]), __ldcg(&w.seg_off[seg]));
  const uint32_t nwords = __ldcg(&w.seg_words[seg]);
  const Glob* g = w.glob;
  const unsigned long long off_bits = __ldcg(&g->off_bits), off_chunks = __ldcg(&g->off_chunks);
  const unsigned long long off_refs = __ldcg(&g->off_refs), off_out = __ldcg(&g->off_out);
  const unsigned long long off_seg = __ldcg(&g->off_seg), off_bitmap = __ldcg(&g->off_bitmap);

  s_code[tid] = __ldcg(&w.tabcode[(size_t)t * 256 + tid]);
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    s_bm[tid] = wi < sh.nw ? __ldcg(&w.bitmap[(size_t)t * sh.nw + wi]) : 0u;
  }
  for (uint32_t i = tid; i < nwords; i += 256) s_bits[i] = 0u;
  __syncthreads();

  // pass 1: bits per literal row; the codes stay in registers
  constexpr int kIters = G::kRowsPerWarp / G::kRPS;
  uint32_t wv[kIters * G::kSPR];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int r = warp * G::kRowsPerWarp + it * G::kRPS + lane / G::kLPR;
    const int64_t b = row0 + r;
    const bool lit = b < B && !((s_bm[r >> 5] >> (r & 31)) & 1u);
    uint32_t nb = 0;
#pragma unroll
    for (int j = 0; j < G::kSPR; ++j) {
      const int d = (lane % G::kLPR) * 4 + j * 128;
      const uint32_t v = lit ? *reinterpret_cast<const uint32_t*>(symt + (size_t)b * D + d) : 0u;
      wv[it * G::kSPR + j] = v;
      nb += (s_code[v & 0xffu] & 0xffu) + (s_code[(v >> 8) & 0xffu] & 0xffu) +
            (s_code[(v >> 16) & 0xffu] & 0xffu) + (s_code[v >> 24] & 0xffu);
    }
#pragma unroll
    for (int off = G::kLPR / 2; off > 0; off >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, off);
    if ((lane % G::kLPR) == 0) s_rowoff[r] = lit ? nb : 0u;
  }
  __syncthreads();

  // row scan: bit offsets, literal ranks, match ranks, outlier offsets
  constexpr int kRPT = (G::kSB + 255) / 256;   // rows per thread
  {
    uint4 loc[kRPT];
    uint4 sum = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const int r = tid * kRPT + k;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G::kSB) {
        const int64_t b = row0 + r;
        if (b < B) {
          const bool m = (s_bm[r >> 5] >> (r & 31)) & 1u;
          v = make_uint4(s_rowoff[r], m ? 0u : 1u, m ? 1u : 0u, m ? 0u : __ldcg(&w.vnout[(size_t)t * B + b]));
        }
      }
      loc[k] = sum;
      sum = add4(sum, v);
    }
    uint4 tot;
    const uint4 ex = block_excl_scan4(sum, &tot, s_warp);
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const int r = tid * kRPT + k;
      if (r < G::kSB) {
        const uint4 p = add4(ex, loc[k]);
        const int64_t b = row0 + r;
        const bool valid = b < B;
        const bool m = (s_bm[r >> 5] >> (r & 31)) & 1u;
        s_rowoff[r] = p.x;
        if (valid && !m) s_litrow[p.y] = (uint16_t)r;
        s_aux[r] = m ? p.z : p.w;
      }
    }
    if (tid == 0) s_segbits = tot.x;
  }
  __syncthreads();

  // pass 2: codes into the shared bitstream
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int r = warp * G::kRowsPerWarp + it * G::kRPS + lane / G::kLPR;
    const int64_t b = row0 + r;
    const bool lit = b < B && !((s_bm[r >> 5] >> (r & 31)) & 1u);
    uint32_t p = s_rowoff[r];
#pragma unroll
    for (int j = 0; j < G::kSPR; ++j) {
      const uint32_t v = wv[it * G::kSPR + j];
      const uint32_t e0 = s_code[v & 0xffu], e1 = s_code[(v >> 8) & 0xffu];
      const uint32_t e2 = s_code[(v >> 16) & 0xffu], e3 = s_code[v >> 24];
      const uint32_t nb = lit ? (e0 & 0xffu) + (e1 & 0xffu) + (e2 & 0xffu) + (e3 & 0xffu) : 0u;
      // exclusive prefix of nb within the row's lane group (stream order = d order)
      uint32_t inc = nb;
#pragma unroll
      for (int off = 1; off < G::kLPR; off <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, inc, off);
        if ((lane % G::kLPR) >= off) inc += n;
      }
      const uint32_t slab_total = __shfl_sync(0xffffffffu, inc, (lane & ~(G::kLPR - 1)) + G::kLPR - 1);
      if (lit) {
        uint32_t q = p + inc - nb;
        put_bits(s_bits, q, e0 >> 8, e0 & 0xffu); q += e0 & 0xffu;
        put_bits(s_bits, q, e1 >> 8, e1 & 0xffu); q += e1 & 0xffu;
        put_bits(s_bits, q, e2 >> 8, e2 & 0xffu); q += e2 & 0xffu;
        put_bits(s_bits, q, e3 >> 8, e3 & 0xffu);
      }
      p += slab_total;
    }
  }
  __syncthreads();

  // bitstream words (16-byte stores; segments start on 128-bit boundaries)
  {
    uint4* dst = reinterpret_cast<uint4*>(out + off_bits + 4ull * base.x);
    const uint4* src = reinterpret_cast<const uint4*>(s_bits);
    for (uint32_t i = tid; i < nwords / 4; i += 256) dst[i] = src[i];
  }
  const uint32_t nlit = __ldcg(&w.seg_cnt[seg]).x;
  // chunk bit lengths
  for (uint32_t k = tid * G::kKC; k < nlit; k += 256 * G::kKC) {
    const uint32_t start = s_rowoff[s_litrow[k]];
    const uint32_t end = k + G::kKC < nlit ? s_rowoff[s_litrow[k + G::kKC]] : s_segbits;
    *reinterpret_cast<uint16_t*>(out + off_chunks + 2ull * (base.y + k / G::kKC)) = (uint16_t)(end - start);
  }
  // references, outliers
  for (int r = tid; r < G::kSB; r += 256) {
    const int64_t b = row0 + r;
    if (b >= B) break;
    const bool m = (s_bm[r >> 5] >> (r & 31)) & 1u;
    if (m) {
      const uint32_t ref = __ldcg(&w.ref[(size_t)t * B + b]);
      const unsigned long long o = off_refs + (unsigned long long)sh.ref_bytes * (base.z + s_aux[r]);
      if (sh.ref_bytes == 2) *reinterpret_cast<uint16_t*>(out + o) = (uint16_t)ref;
      else *reinterpret_cast<uint32_t*>(out + o) = ref;
    } else if (__ldcg(&w.vnout[(size_t)t * B + b]) != 0u) {
      uint32_t k = base.w + s_aux[r];
      const uint8_t* sv = symt + (size_t)b * D;
      const float* xv = x + ((size_t)b * T + t) * D;
      for (int d = 0; d < D; ++d)
        if (sv[d] == 0) *reinterpret_cast<uint32_t*>(out + off_out + 4ull * k++) = __float_as_uint(xv[d]);
    }
  }
  // segment record and bitmap words
  if (tid == 0) {
    uint32_t* rec = reinterpret_cast<uint32_t*>(out + off_seg + (unsigned long long)seg * kSegRecBytes);
    rec[0] = base.x; rec[1] = base.y; rec[2] = base.z; rec[3] = base.w;
  }
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    if (wi < sh.nw)
      *reinterpret_cast<uint32_t*>(out + off_bitmap + 4ull * ((size_t)t * sh.nw + wi)) = s_bm[tid];
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D>
static void launch_compress_d(const float* x, const Shape& sh, const EbParams& ep, const Work& w, uint8_t* out,
                              unsigned long long cap, unsigned long long* out_bytes, uint32_t epoch, cudaStream_t st,
                              Prof* prof) {
  const unsigned grid = (unsigned)(sh.T * sh.nseg);
  if (grid) {
    prof_begin(prof, "k_quantize", st);
    k_quantize<D><<<grid, 256, 0, st>>>(x, sh, ep, w);
    prof_end(prof, st);
    prof_begin(prof, "k_resolve", st);
    k_resolve<D><<<grid, 256, 0, st>>>(x, sh, w);
    prof_end(prof, st);
  }
  prof_begin(prof, "k_codebook", st);
  k_codebook<<<sh.T > 0 ? sh.T : 1, 256, 0, st>>>(sh, ep, w, out, cap, out_bytes, epoch);
  prof_end(prof, st);
  if (grid) {
    prof_begin(prof, "k_emit", st);
    k_emit<D><<<grid, 256, Geo<D>::kSegSyms * 3, st>>>(x, sh, w, out, epoch);
    prof_end(prof, st);
  }
}

cudaError_t launch_compress(const float* x, const Shape& sh, const EbParams& ep, const Work& w, uint8_t* out,
                            unsigned long long cap, unsigned long long* out_bytes, uint32_t epoch, cudaStream_t st,
                            Prof* prof) {
  switch (sh.D) {
    case 4: launch_compress_d<4>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 8: launch_compress_d<8>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 16: launch_compress_d<16>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 32: launch_compress_d<32>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 64: launch_compress_d<64>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 128: launch_compress_d<128>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 256: launch_compress_d<256>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    case 512: launch_compress_d<512>(x, sh, ep, w, out, cap, out_bytes, epoch, st, prof); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int D>
static cudaError_t set_emit_smem() {
  // worst-case bitstream of one segment: every code 24 bits
  return cudaFuncSetAttribute(k_emit<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<D>::kSegSyms * 3);
}

cudaError_t set_kernel_attributes() {
  cudaError_t e = cudaSuccess;
  cudaError_t r[] = {set_emit_smem<4>(), set_emit_smem<8>(), set_emit_smem<16>(), set_emit_smem<32>(),
                     set_emit_smem<64>(), set_emit_smem<128>(), set_emit_smem<256>(), set_emit_smem<512>()};
  for (cudaError_t v : r)
    if (v != cudaSuccess) e = v;
  return e;
}

}  // namespace ebc
