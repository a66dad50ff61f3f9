// ebc_decompress.cu -- decompression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (Huffman and vector-based LZ decoding, dequantization) and §III-E
// ("parallel decompression" of chunks; one or several containers, one per
// batch slice, decoded in the same pass).  The unit is a table of one
// container.  Two launches, no pass over the container before them:
//   k_dec_lit    CTAs per unit: one per group of consecutive segments (more when
//                the unit is decoded in shares, see below).  The
//                sections it reads first sit at offsets that follow from the
//                shape, so the header, the unit's code lengths, the group's
//                segment records and match bitmap are all loaded at once (the
//                header check confirms those offsets; the last CTA also checks
//                every container's header in order and reports the first
//                failure, as the in-order decode does), then the chunk lengths
//                and the group's bitstream (staged in shared memory when it
//                fits).  The CTA builds the unit's canonical decode tables,
//                the literal rows and chunk start bits of its segments, and
//                its warps decode 32 chunks at a time (one per lane; codes,
//                inline outliers), 32 values per lane into a shared-memory
//                slot, stored by the warp with coalesced 16-byte stores.  The
//                last CTA of a unit checks the unit's counts against its table
//                record (and resolves the reference chains of a windowed
//                container); the last unit of a container checks the
//                container's outlier count.
//                When a chunk is one row, a unit has at most kDecShareMaxSeg
//                segments and more CTAs are resident at once than there are
//                groups, each unit gets the resident CTAs divided among the
//                units, and CTA k decodes the k-th of that many
//                equal shares of the unit's chunks (its literal rows and chunk
//                start bits from the segments the share spans), not its group's:
//                the batch's first rows hold most first occurrences, so groups
//                of segments hold very uneven numbers of chunks.  The group
//                checks stay with the groups.
//   k_dec_match  persistent warps take the batch's 32-row bitmap words in turn
//                and copy each matched row from its reference row (the literal
//                it names, or the literal root of its chain).
// Every read of the container is bounds-checked; a failed check records
// EBC_ERR_CORRUPT and stops the remaining work without out-of-bounds access.
#include <cstdint>
#include <type_traits>

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

// Container r of the input: its bounds checked, then its header.
__device__ int container_layout(const uint8_t* in, unsigned long long in_bytes, const unsigned long long* offs,
                                const Shape& sh, int r, Layout* L) {
  const unsigned long long lo = offs ? offs[r] : 0ull, hi = offs ? offs[r + 1] : in_bytes;
  if ((lo & 15ull) != 0ull || lo > hi || hi > in_bytes) return EBC_ERR_CORRUPT;
  uint4 hdr[kHeaderBytes / 16];   // the header, by independent 16-byte loads
  if (hi - lo >= kHeaderBytes) {
#pragma unroll
    for (int k = 0; k < (int)(kHeaderBytes / 16); ++k) hdr[k] = reinterpret_cast<const uint4*>(in + lo)[k];
  }
  const int code = parse_header(reinterpret_cast<const uint8_t*>(hdr), hi - lo,
                                (unsigned long long)slice_rows(sh, r), sh, L);
  L->base = lo;
  L->row0 = (unsigned long long)slice_row0(sh, r);
  return code;
}

// Every container's header (also those without units), one window for all of
// them; writes the call's totals to the status block.  Run once per call (by
// one thread); kept out of line so that its header copies do not raise the
// register count of the decoder's hot loop.  code: the caller's own check so
// far.  first: if not null, receives container 0's layout.
__device__ __noinline__ int check_all_headers(const uint8_t* in, unsigned long long in_bytes,
                                              const unsigned long long* offs, const Shape& sh, Glob* g, int code,
                                              Layout* first) {
  unsigned long long tot[6] = {0, 0, 0, 0, 0, 0};
  uint32_t win0 = 0;
  for (int c = 0; c < sh.R && code == EBC_OK; ++c) {
    Layout Lc{};
    code = container_layout(in, in_bytes, offs, sh, c, &Lc);
    if (c == 0) win0 = Lc.window;
    else if (code == EBC_OK && Lc.window != win0) code = EBC_ERR_CORRUPT;
    tot[0] += Lc.n_lit; tot[1] += Lc.n_match; tot[2] += Lc.n_out; tot[3] += Lc.n_chunks;
    tot[4] += Lc.total; tot[5] += Lc.words;
    if (c == 0 && first) *first = Lc;
  }
  if (code == EBC_OK) {
    g->n_lit = tot[0]; g->n_match = tot[1]; g->n_out = tot[2]; g->n_chunks = tot[3]; g->total = tot[4];
    g->words = tot[5];
    g->window = win0;
  }
  return code;
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

// Canonical ranks over a CTA of kNT threads: thread tid holds the code lengths
// of symbols k * kNT + tid (k < kPer); rank[k] is the number of symbols of the
// same length with a smaller index (in its warp from a match mask, in the
// warps and rounds before from counts).  s_wcnt: (kNT / 32) x (kLmax + 1)
// words, s_run: kLmax + 1 words of shared scratch.
template <int kPer, int kNT>
__device__ void ranks_by_length(const uint32_t (&len)[kPer], uint32_t (&rank)[kPer], uint32_t* s_wcnt,
                                uint32_t* s_run) {
  constexpr int kL = kLmax + 1, kNW = kNT / 32;
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  if (tid < kL) s_run[tid] = 0u;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    for (int i = tid; i < kNW * kL; i += kNT) s_wcnt[i] = 0u;
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
      for (int j = 0; j < kNW; ++j) add += s_wcnt[j * kL + tid];
      s_run[tid] += add;
    }
    __syncthreads();   // the counts are read before the next round clears them
  }
}

// Geometry of the literal decoder.  A CTA takes kSPC consecutive segments of
// one unit (at least 320 rows) and decodes their chunks, a warp taking 32 of
// them at a time (one per lane).  A lane decodes its chunk in pieces of kPiece
// values (a row, or 32 values -- one 128-byte line -- of a longer row) into its
// own shared-memory slot; the warp then stores the 32 pieces with coalesced
// 16-byte stores.  Within a slot, float4 k of lane i sits at k ^ (i mod
// kPieceQ), so that neither the decoding writes nor the storing reads conflict
// on shared-memory banks.
template <int D>
struct DGeo {
  static constexpr int kSB = Geo<D>::kSB;
  static constexpr int kKC = Geo<D>::kKC;
  static constexpr int kSPC = 320 / kSB < 1 ? 1 : 320 / kSB;         // segments per CTA
  static constexpr int kRows = kSPC * kSB;                            // rows per CTA
  static constexpr int kMaxChunks = kRows / kKC;                      // chunks per CTA at most
  static constexpr int kThreads = 128;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kPiece = D < 32 ? D : 32;                      // values per piece
  static constexpr int kPieceQ = kPiece / 4;                          // float4 per piece
  static constexpr int kPiecesPerRow = D / kPiece;
  static constexpr int kBmWords = kSB / 32;                           // bitmap words per segment
  static constexpr int kSegChunks = kSB / kKC;                        // chunks per segment at most
  static constexpr int kSlotQ = kWarps * 32 * kPieceQ;                // float4 of the warps' slots
  static constexpr int kWarpWords = 768;                              // bitstream words staged per warp
};

// A code longer than the first-level table, from the next 32 bits of the
// stream (peek, MSB first).  With canonical codes the codes of each length are
// consecutive and every shorter code sorts before every longer one, so with
// the limits lim[l] = (first[l] + count[l]) << (24 - l) (codes left-aligned to
// 24 bits, non-decreasing in l) the code's length is 12 plus the number of
// lengths l = 12..24 with lim[l] <= the stream's first 24 bits; 25 means no code
// (*bad, and *len = 1).  Returns the symbol.
template <int W>
__device__ __forceinline__ uint32_t long_code(uint32_t peek, const uint32_t* s_lim, const uint32_t* s_first,
                                              const uint32_t* s_offset, const uint16_t* s_sorted, uint32_t* len,
                                              bool* bad) {
  const uint32_t p24 = peek >> (32 - kLmax);
  uint32_t l = kLutBits + 1;
#pragma unroll
  for (int k = kLutBits + 1; k <= kLmax; ++k) l += p24 >= s_lim[k] ? 1u : 0u;
  if (l > (uint32_t)kLmax) {
    *bad = true;
    *len = 1u;
    return 1u;
  }
  *len = l;
  return s_sorted[s_offset[l] + (p24 >> (kLmax - l)) - s_first[l]];
}

// Chunks a warp of the decoder takes at a time: 32, or an even share of a
// group's chunks over its warps when that is fewer.
__device__ __forceinline__ uint32_t batch_chunks(uint32_t nchunks, int warps) {
  const uint32_t share = (nchunks + (uint32_t)warps - 1u) / (uint32_t)warps;
  return share < 1u ? 1u : (share > 32u ? 32u : share);
}

// Units of at most this many segments (of one-row chunks) are decoded in equal
// shares of their chunks.
constexpr int kDecShareMaxSeg = 512;

// ---------------------------------------------------------------------------
// k_dec_lit: grid U * nshare (nshare >= the groups of kSPC segments per unit),
// 128 threads.
// ---------------------------------------------------------------------------
template <int D, int W>
__global__ void __launch_bounds__(128, 5) k_dec_lit(const uint8_t* __restrict__ in, unsigned long long in_bytes,
                                                    const unsigned long long* __restrict__ offs, Shape sh, Work w,
                                                    float* __restrict__ xhat, uint32_t epoch, int nshare) {
  pdl_enter();
  using G = DGeo<D>;
  constexpr int kA = Alph<W>::kA, kNT = G::kThreads;
  constexpr int kLenShift = Alph<W>::kLenShift;
  constexpr uint32_t kSymMask = (1u << kLenShift) - 1u;
  __shared__ __align__(16) uint16_t s_lut[1 << kLutBits];
  __shared__ uint16_t s_sorted[kA];
  __shared__ uint32_t s_first[kLmax + 1], s_offset[kLmax + 1], s_lim[kLmax + 1];
  __shared__ uint32_t s_recs[(G::kSPC + 1) * 4];      // the group's segment records and the one after
  __shared__ uint32_t s_bm[G::kSPC * G::kBmWords];    // the group's match bitmap words
  __shared__ uint16_t s_clen[G::kMaxChunks];          // the group's chunk lengths
  __shared__ uint32_t s_cbit[G::kMaxChunks];          // chunk start bit, from the group's first word
  __shared__ uint32_t s_cinfo[G::kMaxChunks];         // segment in group << 24 | rows << 16 | first rank
  __shared__ uint16_t s_litrow[G::kRows];             // by segment in group, literal rank: row of the segment
  __shared__ __align__(16) float4 s_slot[G::kSlotQ];  // the warps' slots: [kWarps][32 * kPieceQ]
  __shared__ __align__(16) uint32_t s_ws[G::kWarps][G::kWarpWords];   // each warp's batch of bitstream words
  __shared__ uint32_t s_grp[4];                       // chunks, first chunk, first word, words of the group
  __shared__ Layout s_L;
  __shared__ int s_code, s_last;
  __shared__ uint32_t s_cnt[3];                       // literals, matches, outliers of the CTA
  __shared__ uint32_t s_next;                         // next batch of 32 chunks
  __shared__ uint32_t s_rec[4];                       // the unit's table record head: eb, lit, match, out
  __shared__ uint32_t s_len[kA / 4];                  // the unit's code lengths (a byte each)
  __shared__ int s_tbad;                              // the code lengths or the bound are unusable
  __shared__ uint32_t s_count[kLmax + 1], s_wcnt[(kNT / 32) * (kLmax + 1)], s_run[kLmax + 1];
  // decode shares (a chunk is one row, at most kMaxSegU segments per unit): the unit's segment chunk
  // bases and its end, the share's chunk lengths from its first segment's first chunk, and
  // {c0, c1, first segment, last segment, first segment's word, unusable}
  constexpr bool kShareD = G::kKC == 1;
  constexpr int kMaxSegU = kDecShareMaxSeg;
  __shared__ uint32_t s_ucb[kShareD ? kMaxSegU + 1 : 1];
  __shared__ uint16_t s_sclen[kShareD ? G::kMaxChunks + G::kSegChunks : 1];
  __shared__ uint32_t s_sh[6];
  Glob* g = w.glob;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = sh.T;
  // nshare CTAs per unit (at least one per group of kSPC segments; more when the unit's chunks are
  // decoded in shares, CTAs past the groups then only decode)
  const int ngrp = nshare;
  // CTAs go unit-fastest, so the CTAs running at a time write whole rows of the output
  const int nu = sh.U > 0 ? sh.U : 1;
  const int grp = (int)blockIdx.x / nu;
  const int u = (int)blockIdx.x - grp * nu;           // unit: slice u / T, table u % T
  const bool have_unit = u < sh.U;
  const int r = have_unit ? u / T : 0;
  const int t = have_unit ? u - r * T : 0;

  // ---- one round of loads: header, code lengths, segment records, bitmap words, at the offsets the
  //      shape gives (loads outside the container are skipped; its header then fails the check) ----
  const unsigned long long lo = offs ? offs[r] : 0ull, hi = offs ? offs[r + 1] : in_bytes;
  const bool span = (lo & 15ull) == 0ull && lo <= hi && hi <= in_bytes;
  const unsigned long long size = span ? hi - lo : 0ull;
  const uint8_t* cin = in + lo;
  const int64_t nr = slice_rows(sh, r);
  const unsigned int nseg_r = (unsigned int)div_up(nr, G::kSB), nw_r = (unsigned int)div_up(nr, 32);
  const unsigned long long off_seg = kHeaderBytes + (unsigned long long)T * table_rec_bytes(sh.A);
  const unsigned long long off_bm = off_seg + (unsigned long long)T * nseg_r * kSegRecBytes;
  const int s0 = grp * G::kSPC;                                             // first segment of the group
  const int nsg = have_unit ? max(0, min(G::kSPC, (int)nseg_r - s0)) : 0;   // its segments in this slice
  const unsigned long long rec0 = (unsigned long long)t * nseg_r + s0;       // record of its first segment
  const bool rec_end = rec0 + nsg == (unsigned long long)T * nseg_r;         // its last is the container's last
  // (shares only when they add CTAs: with as many CTAs as groups, the groups' own chunks decode sooner)
  const bool use_share = kShareD && have_unit && nseg_r <= (unsigned)kMaxSegU && ngrp > div_up(sh.nseg, G::kSPC);
  if (use_share) {   // the unit's segment chunk bases (record word 1), and the next table's first
    const unsigned int nb = nseg_r + (t + 1 < T ? 1u : 0u);
    for (unsigned int i = tid; i < nb; i += kNT) {
      const unsigned long long o = off_seg + ((unsigned long long)t * nseg_r + i) * kSegRecBytes + 4ull;
      s_ucb[i] = o + 4 <= size ? ld32(cin + o) : 0u;
    }
  }
  if (have_unit) {
    const uint8_t* rec = cin + kHeaderBytes + (size_t)t * Alph<W>::kRecBytes;
    const bool rec_in = kHeaderBytes + (unsigned long long)(t + 1) * Alph<W>::kRecBytes <= size;
    if (tid < 4) s_rec[tid] = rec_in ? ld32(rec + 4 * tid) : 0u;
    for (int i = tid; i < kA / 4; i += kNT) s_len[i] = rec_in ? ld32(rec + 16 + 4 * i) : 0u;
    const int nrw = 4 * (nsg + (rec_end ? 0 : 1));
    for (int i = tid; i < nrw; i += kNT) {
      const unsigned long long o = off_seg + rec0 * kSegRecBytes + 4ull * i;
      s_recs[i] = o + 4 <= size ? ld32(cin + o) : 0u;
    }
    for (int i = tid; i < nsg * G::kBmWords; i += kNT) {
      const unsigned long long wi = (unsigned long long)s0 * G::kBmWords + i;   // word of the unit's bitmap
      const unsigned long long o = off_bm + 4ull * ((unsigned long long)t * nw_r + wi);
      s_bm[i] = wi < nw_r && o + 4 <= size ? ld32(cin + o) : 0u;
    }
  }
  for (int i = tid; i < (1 << kLutBits) / 8; i += kNT) reinterpret_cast<uint4*>(s_lut)[i] = make_uint4(0, 0, 0, 0);
  if (tid <= kLmax) s_count[tid] = 0u;
  if (tid == 0) {
    s_tbad = 0;
    // the grid's last CTA (the batch's last rows: mostly matches, little to decode) checks the
    // containers in order and reports the first failure (the code the in-order decode of the
    // containers meets first); a CTA whose own container fails stops silently (code -1) and only takes
    // part in the unit's counters
    if (blockIdx.x == gridDim.x - 1) {
      const int all = check_all_headers(in, in_bytes, offs, sh, g, EBC_OK, nullptr);
      if (all != EBC_OK) dec_fail(g, epoch, all);
    }
    Layout L{};
    const int code = have_unit ? (container_layout(in, in_bytes, offs, sh, r, &L) == EBC_OK ? EBC_OK : -1) : EBC_OK;
    if (have_unit && t == 0 && grp == 0 && code == EBC_OK) w.lay[r] = L;   // for the match copy
    if (use_share && t + 1 == T) s_ucb[nseg_r] = code == EBC_OK && L.n_chunks < 0xFFFFFFFFull ? (uint32_t)L.n_chunks : 0u;
    s_L = L;
    s_code = code;
    s_cnt[0] = s_cnt[1] = s_cnt[2] = 0u;
    s_grp[0] = 0u;
    if (tid == 0 && code == EBC_OK && have_unit) {
      // the group's chunk and word ranges, from its first record and the one after its last
      const uint32_t cb0 = nsg > 0 ? s_recs[1] : 0u, wb0 = nsg > 0 ? s_recs[0] : 0u;
      const unsigned long long cb1 = nsg == 0 ? cb0 : (rec_end ? L.n_chunks : s_recs[4 * nsg + 1]);
      const unsigned long long wb1 = nsg == 0 ? wb0 : (rec_end ? L.words : s_recs[4 * nsg]);
      // (chunks hold literal rows, at least one bit per code: a group with chunks has words)
      if (cb1 < cb0 || cb1 > L.n_chunks || cb1 - cb0 > (unsigned long long)G::kMaxChunks || wb1 < wb0 ||
          wb1 > L.words || (wb0 & 3u) || (wb1 & 3ull) || (cb1 > cb0 && wb1 == wb0)) {
        s_code = EBC_ERR_CORRUPT;
      } else {
        s_grp[0] = (uint32_t)(cb1 - cb0);
        s_grp[1] = cb0;
        s_grp[2] = wb0;
        s_grp[3] = (uint32_t)(wb1 - wb0);
      }
    }
    s_next = (uint32_t)G::kWarps * batch_chunks(s_grp[0], G::kWarps);
  }
  __syncthreads();
  const Layout& L = s_L;   // read from shared memory where used

  // whether the tables are built: read once here (s_code changes only after the barriers below)
  const bool build = s_code == EBC_OK && have_unit;

  // ---- decode share (with a chunk per row and a unit of at most kMaxSegU segments): this CTA decodes
  //      the grp-th of ngrp equal shares of its unit's chunks instead of its group's chunks (the batch's
  //      first rows hold most first occurrences, so groups hold very uneven numbers of chunks).  Its
  //      range and first segments are found now and their loads issued into registers, so that they
  //      are in flight while the tables are built and the group is checked ----
  const bool share = build && use_share;   // (uniform: s_code was read after the barrier)
  constexpr int kLenPer = (G::kMaxChunks + G::kSegChunks + kNT - 1) / kNT;   // chunk lengths per thread
  uint32_t c0 = 0, c1 = 0, sa = 0, sb = 0, cbS = 0;
  bool sbad = false;
  uint32_t pre_len[kLenPer], pre_wbS = 0, pre_word = 0, pre_bm = 0;
  if (share) {
    if (tid == 0) {
      const uint32_t u0 = s_ucb[0], u1 = s_ucb[nseg_r];
      uint32_t a0 = u0, a1 = u0, unusable = u1 < u0 || u1 > L.n_chunks;
      if (!unusable) {
        const unsigned long long n_u = u1 - u0;
        a0 = u0 + (uint32_t)(n_u * (unsigned)grp / (unsigned)ngrp);
        a1 = u0 + (uint32_t)(n_u * (unsigned)(grp + 1) / (unsigned)ngrp);
        unusable = a1 - a0 > (uint32_t)G::kMaxChunks;
      }
      s_sh[0] = a0;
      s_sh[1] = a1;
      s_sh[2] = s_sh[3] = 0xFFFFFFFFu;
      s_sh[5] = unusable;
    }
    __syncthreads();
    c0 = s_sh[0];
    c1 = s_sh[1];
    if (c1 > c0 && !s_sh[5]) {   // the segments holding chunks c0 and c1 - 1
      for (unsigned int sg = tid; sg < nseg_r; sg += kNT) {
        const uint32_t a = s_ucb[sg], e = s_ucb[sg + 1];
        if (a <= c0 && c0 < e) s_sh[2] = sg;
        if (a <= c1 - 1u && c1 - 1u < e) s_sh[3] = sg;
      }
    }
    __syncthreads();
    sa = s_sh[2];
    sb = s_sh[3];
    // (an inconsistent share exists only in a corrupt container, whose group checks fail elsewhere)
    sbad = c1 > c0 && (s_sh[5] != 0u || sa >= nseg_r || sb >= nseg_r || sb < sa);
    cbS = c1 > c0 && !sbad ? s_ucb[sa] : c0;   // the first chunk of the first segment
    if (c1 - cbS > (uint32_t)(G::kMaxChunks + G::kSegChunks)) sbad = true;
    if (c1 > c0 && !sbad) {
      // the chunk lengths from cbS to c1, the first segment's first word, and each warp's first
      // segment's first word and bitmap words
      const uint16_t* cl = reinterpret_cast<const uint16_t*>(cin + L.off_chunks);
#pragma unroll
      for (int k = 0; k < kLenPer; ++k) {
        const uint32_t i = (uint32_t)(k * kNT + tid);
        pre_len[k] = i < c1 - cbS ? (uint32_t)cl[cbS + i] : 0u;
      }
      if (tid == 0) pre_wbS = ld32(cin + off_seg + ((unsigned long long)t * nseg_r + sa) * kSegRecBytes);
      const uint32_t sg = sa + (uint32_t)warp;
      if (sg <= sb) {
        if (lane == 0) pre_word = ld32(cin + off_seg + ((unsigned long long)t * nseg_r + sg) * kSegRecBytes);
        const int64_t nv = nr - ((int64_t)sg * G::kSB + (int64_t)lane * 32);
        const unsigned long long bwi = (unsigned long long)sg * G::kBmWords + lane;
        const unsigned long long o = off_bm + 4ull * ((unsigned long long)t * nw_r + bwi);
        if (lane < G::kBmWords && nv > 0 && bwi < nw_r && o + 4 <= size) pre_bm = ld32(cin + o);
      }
    } else {
#pragma unroll
      for (int k = 0; k < kLenPer; ++k) pre_len[k] = 0u;
    }
  }
  // ---- second round: the chunk lengths (in flight while the tables are built) ----
  if (build) {
    const uint16_t* cl = reinterpret_cast<const uint16_t*>(cin + L.off_chunks) + s_grp[1];
    for (uint32_t i = tid; i < s_grp[0]; i += kNT) s_clen[i] = cl[i];
  }

  // ---- the unit's canonical decode tables, from its code lengths: lengths at most 24, a Kraft sum of
  //      at most 1 and a usable bound, else the container is corrupt ----
  if (build) {
    bool bad = false;
    for (int i = tid; i < kA; i += kNT) {
      const uint32_t len = (s_len[i >> 2] >> (8 * (i & 3))) & 0xffu;
      if (len > (uint32_t)kLmax) bad = true;
      else if (len) atomicAdd(&s_count[len], 1u);
    }
    if (bad) s_tbad = 1;   // (benign race: any writer stores the same value)
    __syncthreads();
    if (tid < 32) {
      // lane l (1..24): the Kraft term of length l, the first canonical code of length l (sum over
      // k < l of count[k] << (l - k)), its offset in sorted[] (the counts below l), and the limit
      // (first + count) << (24 - l) of the long-code search
      const int l = lane;
      const uint32_t cnt = l >= 1 && l <= kLmax ? s_count[l] : 0u;
      unsigned long long kraft = l >= 1 && l <= kLmax ? (unsigned long long)cnt << (kLmax - l) : 0ull;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kraft += __shfl_xor_sync(0xffffffffu, kraft, off);
      unsigned long long first = 0;
      uint32_t below = 0;
      for (int k = 1; k < l && k <= kLmax; ++k) {
        first += (unsigned long long)s_count[k] << (l - k);
        below += s_count[k];
      }
      if (l <= kLmax) {
        s_first[l] = l ? (uint32_t)first : 0u;
        s_offset[l] = l ? below : 0u;
        // (a Kraft sum of at most 1 keeps first + count <= 2^l: the limit fits 25 bits)
        s_lim[l] = l ? (uint32_t)((first + cnt) << (kLmax - l)) : 0u;
      }
      if (lane == 0 && (kraft > (1ull << kLmax) || !eb_usable(__uint_as_float(s_rec[0])))) s_tbad = 1;
    }
    __syncthreads();
    if (!s_tbad) {
      // each symbol's rank among the symbols of its length below it: its index in sorted[] is
      // offset[len] + rank, its code first[len] + rank
      constexpr int kPer = kA / kNT;
      constexpr int kLenShiftT = Alph<W>::kLenShift;
      uint32_t lens[kPer], rk[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = k * kNT + tid;
        lens[k] = (s_len[i >> 2] >> (8 * (i & 3))) & 0xffu;
      }
      ranks_by_length<kPer, kNT>(lens, rk, s_wcnt, s_run);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const uint32_t len = lens[k], i = (uint32_t)(k * kNT + tid);
        if (!len) continue;
        s_sorted[s_offset[len] + rk[k]] = (uint16_t)i;
        if (len <= (uint32_t)kLutBits) {
          const uint32_t code = s_first[len] + rk[k];
          const uint32_t l0 = code << (kLutBits - len), n = 1u << (kLutBits - len);
          const uint16_t e = (uint16_t)(i | (len << kLenShiftT));
          if (n >= 8u) {   // 16-byte aligned runs of 8 entries (l0 is a multiple of n)
            const uint32_t e2 = (uint32_t)e | ((uint32_t)e << 16);
            uint4* p = reinterpret_cast<uint4*>(s_lut + l0);
            for (uint32_t q = 0; q < n / 8u; ++q) p[q] = make_uint4(e2, e2, e2, e2);
          } else {
            for (uint32_t q = 0; q < n; ++q) s_lut[l0 + q] = e;
          }
        }
      }
    }
    if (tid == 0 && s_tbad) s_code = EBC_ERR_CORRUPT;
    __syncthreads();
  }
  bool ok = s_code == EBC_OK && have_unit;

  // ---- the group's segments: literal rows, chunk start bits, chain checks (a warp per segment) ----
  uint32_t nchunks = 0;
  if (ok) {
    const uint32_t cb0 = s_grp[1], wb0 = s_grp[2], ngc = s_grp[0];
    bool bad = false;
    for (int j = warp; j < nsg; j += G::kWarps) {
      const int s = s0 + j;
      const unsigned long long ri = rec0 + j;   // record of the segment
      const uint32_t* rc = s_recs + 4 * j;
      const uint32_t word_off = rc[0], chunk_base = rc[1], match_base = rc[2], nbits = rc[3];
      const bool last = j == nsg - 1 && rec_end;
      const unsigned long long nx_word = last ? L.words : rc[4], nx_chunk = last ? L.n_chunks : rc[5],
                               nx_match = last ? L.n_match : rc[6];
      const int64_t row0 = (int64_t)s * G::kSB;   // within the slice
      // literal rows in row order, two bitmap words per lane at most
      uint32_t nlit = 0, nvalid = 0;
#pragma unroll
      for (int half = 0; half < (G::kBmWords + 31) / 32; ++half) {
        const int wi = half * 32 + lane;
        uint32_t litw = 0, valid = 0;
        if (wi < G::kBmWords) {
          const int64_t nv = nr - (row0 + (int64_t)wi * 32);
          valid = nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
          if (nv > 0) {
            const uint32_t bm = s_bm[j * G::kBmWords + wi];
            if (bm & ~valid) bad = true;   // match bits past the slice
            litw = ~bm & valid;
          }
        }
        uint32_t tot, vt;
        const uint32_t k = nlit + warp_excl(__popc(litw), &tot);
        warp_excl(__popc(valid), &vt);
        // the word's literal rows, by rank: lane b of the warp takes bit b of each word in turn
        const uint32_t wbase = (uint32_t)(half * 32);
        for (int wl = 0; wl < 32; ++wl) {
          const uint32_t lw = __shfl_sync(0xffffffffu, litw, wl), kb = __shfl_sync(0xffffffffu, k, wl);
          if ((lw >> lane) & 1u)
            s_litrow[j * G::kSB + kb + __popc(lw & ((1u << lane) - 1u))] = (uint16_t)((wbase + wl) * 32 + lane);
          if (wbase + wl + 1 >= (uint32_t)G::kBmWords) break;
        }
        nlit += tot;
        nvalid += vt;
      }
      const uint32_t nmatch = nvalid - nlit;
      const uint32_t nch = (nlit + G::kKC - 1) / G::kKC;
      const unsigned long long seg_words = ((nbits + 127ull) >> 7) * 4ull;
      const uint32_t cl0 = chunk_base - cb0;
      bool good = (unsigned long long)chunk_base + nch == nx_chunk && nx_chunk <= L.n_chunks &&
                  (unsigned long long)match_base + nmatch == nx_match && nx_match <= L.n_match &&
                  (unsigned long long)word_off + seg_words == nx_word && nx_word <= L.words &&
                  (ri != 0 || (word_off == 0 && chunk_base == 0 && match_base == 0)) && chunk_base >= cb0 &&
                  cl0 + nch <= ngc && word_off >= wb0;
      if (__all_sync(0xffffffffu, good)) {   // chunk start bits: the segment's first bit + the lengths before
        const uint32_t bit0 = (word_off - wb0) * 32u;   // the segment's first bit in the group's range
        uint32_t acc = 0;
#pragma unroll
        for (int half = 0; half < (G::kSegChunks + 31) / 32; ++half) {
          const uint32_t c = half * 32 + lane;
          const uint32_t len = c < nch ? (uint32_t)s_clen[cl0 + c] : 0u;
          uint32_t tot;
          const uint32_t st = acc + warp_excl(len, &tot);
          if (c < nch) {
            s_cbit[cl0 + c] = bit0 + st;
            s_cinfo[cl0 + c] = ((uint32_t)j << 24) | (min((uint32_t)G::kKC, nlit - c * G::kKC) << 16) |
                               (c * G::kKC);
          }
          acc += tot;
        }
        good = acc == nbits;
        if (lane == 0) {
          atomicAdd(&s_cnt[0], nlit);
          atomicAdd(&s_cnt[1], nmatch);
        }
      }
      if (!__all_sync(0xffffffffu, good)) bad = true;
    }
    if (bad) s_code = EBC_ERR_CORRUPT;
    __syncthreads();
    ok = s_code == EBC_OK;
    nchunks = ok ? s_grp[0] : 0u;
  }

  // ---- decode share, its metadata: a warp per segment of the share, its literal rows by rank and the
  //      chunk start bits ----
  if (share && ok) {
#pragma unroll
    for (int k = 0; k < kLenPer; ++k) {
      const uint32_t i = (uint32_t)(k * kNT + tid);
      if (i < (uint32_t)(G::kMaxChunks + G::kSegChunks)) s_sclen[i] = (uint16_t)pre_len[k];
    }
    if (tid == 0) s_sh[4] = pre_wbS;
    __syncthreads();
    const uint32_t wbS = s_sh[4];
    if (c1 > c0 && !sbad && ((wbS & 3u) || wbS > L.words)) sbad = true;
    if (c1 > c0 && !sbad) {
      const uint32_t below = (1u << lane) - 1u;
      for (uint32_t sg = sa + (uint32_t)warp; sg <= sb; sg += (uint32_t)G::kWarps) {
        const uint32_t a = s_ucb[sg], e = s_ucb[sg + 1];
        if (e <= a) continue;   // no literal rows
        const bool first_seg = sg == sa + (uint32_t)warp;   // its word and bitmap words were loaded early
        const uint32_t word_off = __shfl_sync(
            0xffffffffu,
            first_seg ? pre_word
                      : (lane == 0 ? ld32(cin + off_seg + ((unsigned long long)t * nseg_r + sg) * kSegRecBytes) : 0u),
            0);
        const int64_t row0 = (int64_t)sg * G::kSB;   // within the slice
        // literal rows in row order: rank j is chunk a + j (its row into s_cinfo when in the share)
        uint32_t nlit = 0;
#pragma unroll
        for (int half = 0; half < (G::kBmWords + 31) / 32; ++half) {
          const int wi = half * 32 + lane;
          uint32_t litw = 0;
          if (wi < G::kBmWords) {
            const int64_t nv = nr - (row0 + (int64_t)wi * 32);
            const uint32_t valid = nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
            const unsigned long long bwi = (unsigned long long)sg * G::kBmWords + wi;
            const unsigned long long o = off_bm + 4ull * ((unsigned long long)t * nw_r + bwi);
            const uint32_t bm =
                first_seg && half == 0 ? pre_bm : (nv > 0 && bwi < nw_r && o + 4 <= size ? ld32(cin + o) : 0u);
            litw = ~bm & valid;
          }
          uint32_t tot;
          const uint32_t k = nlit + warp_excl(__popc(litw), &tot);
          const uint32_t wbase = (uint32_t)(half * 32);
          for (int wl = 0; wl < 32; ++wl) {
            const uint32_t lw = __shfl_sync(0xffffffffu, litw, wl), kb = __shfl_sync(0xffffffffu, k, wl);
            if ((lw >> lane) & 1u) {
              const uint32_t c = a + kb + __popc(lw & below);
              if (c >= c0 && c < c1) s_cinfo[c - c0] = (uint32_t)(row0 + (int64_t)((wbase + wl) * 32 + lane));
            }
            if (wbase + wl + 1 >= (uint32_t)G::kBmWords) break;
          }
          nlit += tot;
        }
        if (nlit != e - a) sbad = true;
        // chunk start bits: the segment's first bit (relative to the share's first segment) + the lengths
        // of its chunks before
        uint32_t acc = 0;
#pragma unroll
        for (int half = 0; half < (G::kSegChunks + 31) / 32; ++half) {
          const uint32_t j = (uint32_t)(half * 32 + lane);
          const uint32_t c = a + j;
          const uint32_t len = j < e - a && c < c1 ? (uint32_t)s_sclen[c - cbS] : 0u;
          uint32_t tot;
          const uint32_t st = acc + warp_excl(len, &tot);
          if (j < e - a && c >= c0 && c < c1) {
            s_cbit[c - c0] = (word_off - wbS) * 32u + st;
            s_clen[c - c0] = (uint16_t)len;
          }
          acc += tot;
        }
      }
    }
    if (sbad) s_code = EBC_ERR_CORRUPT;   // (benign race: any writer stores the same value)
    if (tid == 0) {
      s_grp[2] = wbS;
      s_grp[3] = wbS <= L.words ? (uint32_t)(L.words - wbS) : 0u;
      s_next = (uint32_t)G::kWarps * batch_chunks(c1 - c0, G::kWarps);
    }
    __syncthreads();
    ok = s_code == EBC_OK;
    nchunks = ok ? c1 - c0 : 0u;
  }

  // ---- decode: a warp takes 32 chunks at a time, a piece per lane into its slot, then stores them ----
  // Four symbols at a time on a branch-free path that assumes ordinary codes (first-level table,
  // symbol field not 0); when one of the four was an outlier or a longer code, the four are decoded
  // again from the same bit position by the general path.
  uint32_t nout = 0;
  bool bad = false;
  if (ok) {
    const uint32_t gwords = s_grp[3];   // > 0 whenever there are chunks
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(cin + L.off_bits) + s_grp[2];   // the group's words
    const int64_t brow0 = (int64_t)L.row0;
    float4* slot = s_slot + warp * 32 * G::kPieceQ;
    uint32_t* ws = s_ws[warp];
    // the reconstruction fl32((sym - R) * 2 eb): the integer sym - R (|.| < 2^22) becomes a float
    // exactly by placing it in the mantissa of 1.5 * 2^23 and subtracting that
    const float ebx2 = __fmul_rn(2.0f, __uint_as_float(s_rec[0]));
    auto value = [&](uint32_t sym) -> float {
      return __fmul_rn(__fsub_rn(__uint_as_float(0x4B400000u - (uint32_t)Alph<W>::kR + sym), 12582912.0f), ebx2);
    };
    // batches of up to 32 chunks, smaller when the group has few, so that every warp takes a share
    const uint32_t bsz = batch_chunks(nchunks, G::kWarps);
    for (uint32_t b0 = (uint32_t)warp * bsz; b0 < nchunks;) {
      // the batch's words (its chunks are consecutive, so their bits are too): staged in this warp's
      // buffer with coalesced 16-byte loads when they fit, else read from global memory
      const uint32_t clast = min(b0 + bsz - 1u, nchunks - 1u);
      const uint32_t wlo = (s_cbit[b0] >> 5) & ~3u;
      const uint32_t whi = min(((s_cbit[clast] + s_clen[clast]) >> 5) + 3u, gwords);   // exclusive; the window
                                                                                         // reads 2 words ahead
      const bool staged = whi - wlo <= (uint32_t)G::kWarpWords;
      if (staged) {
        const uint32_t n4 = (whi - wlo + 3u) >> 2;   // within the group's words (a multiple of 4)
        const uint4* src = reinterpret_cast<const uint4*>(gw + wlo);
        for (uint32_t i = lane; i < n4; i += 32) reinterpret_cast<uint4*>(ws)[i] = __ldg(src + i);
        __syncwarp();
      }
      const uint32_t nst = whi - wlo;   // staged words (reads past them repeat the last)
      auto run = [&](auto staged_tag) {
        constexpr bool kStaged = decltype(staged_tag)::value;
        auto word = [&](uint32_t i) -> uint32_t {
          if constexpr (kStaged) return ws[min(i - wlo, nst - 1u)];
          else return __ldg(gw + min(i, gwords - 1u));
        };
        const uint32_t c = b0 + lane;
        const bool mine = (uint32_t)lane < bsz && c < nchunks;
        const uint32_t info = mine ? s_cinfo[c] : 0u;
        const uint32_t start = mine ? s_cbit[c] : s_cbit[b0];
        const uint32_t clen = mine ? (uint32_t)s_clen[c] : 0u;
        const int j = (int)(info >> 24);
        // (a share's chunk is one row, which s_cinfo holds; a group's chunk: segment, rows, first rank)
        const uint32_t rows = share ? (mine ? 1u : 0u) : (info >> 16) & 0xffu, first = info & 0xffffu;
        const uint32_t npieces = rows * G::kPiecesPerRow;
        // bit buffer: the next nb bits, left-aligned in buf; wp is the next word to read (reads past the
        // group's words repeat its last word; they never decide a code of a valid chunk)
        const uint32_t wp0 = start >> 5, sbit = start & 31u;
        uint32_t wp = wp0 + 2u, nb = 64u - sbit;
        unsigned long long buf = (((unsigned long long)word(wp0) << 32) | word(wp0 + 1u)) << sbit;
        auto refill = [&]() {   // nb <= 32 before: one more word
          buf |= (unsigned long long)word(wp) << (32u - nb);
          ++wp;
          nb += 32u;
        };
        float* rowdst = nullptr;
        const uint32_t allp = __reduce_max_sync(0xffffffffu, npieces);
        for (uint32_t p = 0; p < allp; ++p) {
          const bool act = p < npieces;
          if (act) {
            const uint32_t rk = p / G::kPiecesPerRow, pc = p % G::kPiecesPerRow;
            if (pc == 0) {
              const int64_t b = share ? brow0 + (int64_t)info
                                      : brow0 + (int64_t)(s0 + j) * G::kSB + s_litrow[j * G::kSB + first + rk];
              rowdst = xhat + ((size_t)b * sh.T_out + sh.t_off + t) * D;
            }
#pragma unroll 1
            for (int q4 = 0; q4 < G::kPieceQ; ++q4) {
              const unsigned long long buf0 = buf;
              const uint32_t nb0 = nb, wq = wp;
              float o[4];
              uint32_t plain = 1u;   // all four are first-table codes of ordinary symbols
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if ((q & 1) == 0 && nb < 22u) refill();   // two first-table codes take at most 22 bits
                const uint32_t e = s_lut[(uint32_t)(buf >> (64 - kLutBits))];
                const uint32_t sym = e & kSymMask;
                plain = sym ? plain : 0u;
                o[q] = value(sym);
                buf <<= e >> kLenShift;
                nb -= e >> kLenShift;
              }
              if (!plain) {   // an outlier or a longer code among the four: decode them again, in general
                buf = buf0;
                nb = nb0;
                wp = wq;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (nb <= 32u) refill();   // at least 33 bits: any code fits
                  const uint32_t peek = (uint32_t)(buf >> 32);
                  const uint32_t e = s_lut[peek >> (32 - kLutBits)];
                  uint32_t sym = e & kSymMask, len = e >> kLenShift;
                  if (sym == 0u && len == 0u)
                    sym = long_code<W>(peek, s_lim, s_first, s_offset, s_sorted, &len, &bad);
                  buf <<= len;
                  nb -= len;
                  float v = value(sym);
                  if (sym == 0u) {   // outlier: the next 32 bits are the raw value
                    if (nb <= 32u) refill();
                    v = __uint_as_float((uint32_t)(buf >> 32));
                    buf <<= 32;
                    nb -= 32u;
                    ++nout;
                  }
                  o[q] = v;
                }
              }
              slot[lane * G::kPieceQ + (q4 ^ (lane & (G::kPieceQ - 1)))] = make_float4(o[0], o[1], o[2], o[3]);
            }
          }
          __syncwarp();
          // the warp's pieces: float4 i of the step goes to piece i / kPieceQ (lane), float4 i % kPieceQ
          const unsigned long long pdst =
              act ? (unsigned long long)(rowdst + (p % G::kPiecesPerRow) * G::kPiece) : 0ull;
#pragma unroll
          for (int k = 0; k < G::kPieceQ; ++k) {
            const int i = k * 32 + lane;
            const int owner = i / G::kPieceQ, q = i % G::kPieceQ;
            const unsigned long long d = __shfl_sync(0xffffffffu, pdst, owner);
            if (d) __stcs(reinterpret_cast<float4*>(d) + q, slot[owner * G::kPieceQ + (q ^ (owner & (G::kPieceQ - 1)))]);
          }
          __syncwarp();
        }
        if (mine && (wp - wp0) * 32u - nb - sbit != clen) bad = true;
      };
      if (staged) run(std::integral_constant<bool, true>{});
      else run(std::integral_constant<bool, false>{});
      __syncwarp();   // the staged words are read before the next batch overwrites them
      // the next batch of 32 chunks of the group
      uint32_t nb = 0;
      if (lane == 0) nb = atomicAdd(&s_next, bsz);
      b0 = __shfl_sync(0xffffffffu, nb, 0);
    }
  }
  if (bad) s_code = EBC_ERR_CORRUPT;   // (benign race: any writer stores the same value)
  nout = __reduce_add_sync(0xffffffffu, nout);
  if (lane == 0 && nout) atomicAdd(&s_cnt[2], nout);
  __syncthreads();
  if (have_unit && s_code > 0 && tid == 0) dec_fail(g, epoch, s_code);

  // ---- the unit's last CTA: its counts against the table record ----
  if (!have_unit) return;
  if (tid == 0) {
    uint4* acc = w.uacc + u;
    if (s_cnt[0]) atomicAdd(&acc->x, s_cnt[0]);
    if (s_cnt[1]) atomicAdd(&acc->y, s_cnt[1]);
    if (s_cnt[2]) atomicAdd(&acc->z, s_cnt[2]);
    __threadfence();
    s_last = atomicAdd(&acc->w, 1u) == (unsigned)ngrp - 1u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const bool checked = !dec_aborted(g, epoch);   // the counts mean something only if nothing failed
  __shared__ uint32_t s_unit[3];
  if (tid == 0) {
    uint4* acc = w.uacc + u;
    s_unit[0] = atomicExch(&acc->x, 0u);
    s_unit[1] = atomicExch(&acc->y, 0u);
    s_unit[2] = atomicExch(&acc->z, 0u);
    atomicExch(&acc->w, 0u);   // clean for the next call
  }
  __syncthreads();
  int fail = EBC_OK;
  if (checked && s_code == EBC_OK) {
    const uint8_t* rec = cin + kHeaderBytes + (size_t)t * Alph<W>::kRecBytes;
    if (ld32(rec + 4) != s_unit[0] || ld32(rec + 8) != s_unit[1] || ld32(rec + 12) != s_unit[2])
      fail = EBC_ERR_CORRUPT;
  }
  if (checked && s_code == EBC_OK && L.window && L.nseg > 0 && fail == EBC_OK) {
    // window references: every row's source (itself for a literal, b - distance for a match),
    // from the unit's bitmap and one-byte distances, resolved to the literal roots of the chains.
    // Rows go in blocks of kBlk: a block's sources are built in shared memory (the staging words
    // are free now), a source in an earlier block is replaced by its final root (the last 256
    // roots of the previous block are kept: a distance is at most 255), then the block's chains
    // are resolved by pointer jumping in shared memory and its roots written out.
    constexpr int kBlk = 2048, kBW = kBlk / 32;
    static_assert(G::kWarps * G::kWarpWords >= kBlk + 256, "block and tail fit the staging words");
    static_assert(kNT >= kBW && kBlk % kNT == 0 && 32 % (kBlk / kNT) == 0,
                  "a thread per bitmap word of the block; each thread's run of rows inside one word");
    __shared__ uint32_t s_wc[kNT / 32], s_bmw[kBW], s_pre[kBW];
    __shared__ int s_wbad;
    uint32_t* s_blk = &s_ws[0][0];        // [kBlk] sources (absolute rows), then roots
    uint32_t* s_tail = s_blk + kBlk;      // roots of the previous block's last 256 rows
    if (tid == 0) s_wbad = 0;
    const int64_t n = (int64_t)L.n, row0 = (int64_t)L.row0;
    const int64_t nw = L.nw;
    const uint32_t* bmt = reinterpret_cast<const uint32_t*>(cin + L.off_bitmap) + (size_t)t * nw;
    const uint8_t* dist = cin + L.off_refs;
    const uint32_t* srec = reinterpret_cast<const uint32_t*>(cin + L.off_seg);
    const unsigned long long mbase = srec[4ull * ((unsigned long long)t * L.nseg) + 2];
    uint32_t* src = w.srcrow + (size_t)t * sh.B + row0;
    unsigned long long carry = 0;   // matches of the unit before the block
    __syncthreads();
    for (int64_t bs = 0; bs < n; bs += kBlk) {
      const int nb = (int)min((int64_t)kBlk, n - bs);
      // the block's bitmap words and the matches before each
      const int64_t wi = bs / 32 + tid;
      const uint32_t bm = (tid < kBW && wi < nw) ? __ldcg(&bmt[wi]) : 0u;
      uint32_t wt;
      const uint32_t ex = warp_excl((uint32_t)__popc(bm), &wt);
      if (lane == 0) s_wc[warp] = wt;
      __syncthreads();
      if (tid < kBW) {
        uint32_t before = 0;
        for (int k = 0; k < warp; ++k) before += s_wc[k];
        s_bmw[tid] = bm;
        s_pre[tid] = before + ex;
      }
      uint32_t blk_matches = 0;
      for (int k = 0; k < kNT / 32; ++k) blk_matches += s_wc[k];
      __syncthreads();
      {   // sources: each thread a run of the block's rows
        constexpr int kRun = kBlk / kNT;
        const int i0 = tid * kRun;
        const int wd = i0 >> 5;
        const uint32_t bmv = s_bmw[wd];
        const unsigned long long rk0 = mbase + carry + s_pre[wd];
#pragma unroll 4
        for (int jj = 0; jj < kRun; ++jj) {
          const int i = i0 + jj;
          if (i >= nb) break;
          const int bit = i & 31;
          const int64_t b = bs + i;   // row of the slice
          uint32_t from = (uint32_t)(row0 + b);
          if ((bmv >> bit) & 1u) {
            const unsigned long long k = rk0 + __popc(bmv & ((1u << bit) - 1u));
            const uint32_t d = k < L.n_match ? dist[k] : 0u;
            if (d == 0u || d > L.window || (int64_t)d > b) {
              s_wbad = 1;
            } else {
              const int64_t sb = b - d;
              from = sb >= bs ? (uint32_t)(row0 + sb) : s_tail[sb - (bs - 256)];   // earlier block: its root
            }
          }
          s_blk[i] = from;
        }
      }
      carry += blk_matches;
      __syncthreads();
      for (int rd = 0; rd < 12; ++rd) {   // chains inside the block are shorter than 2^11
        for (int i = tid; i < nb; i += kNT) {
          const int64_t rel = (int64_t)s_blk[i] - row0 - bs;
          if (rel >= 0 && rel < i) s_blk[i] = s_blk[rel];
        }
        __syncthreads();
      }
      for (int i = tid; i < nb; i += kNT) src[bs + i] = s_blk[i];
      if (nb == kBlk)
        for (int j = tid; j < 256; j += kNT) s_tail[j] = s_blk[kBlk - 256 + j];
      __syncthreads();
    }
    if (s_wbad) fail = EBC_ERR_CORRUPT;
  }
  if (tid == 0) {
    if (fail != EBC_OK) dec_fail(g, epoch, fail);
    // the container's outliers: the last of its T units compares their sum with the header
    uint2* cacc = w.cacc + r;
    atomicAdd(&cacc->x, s_unit[2]);
    __threadfence();
    if (atomicAdd(&cacc->y, 1u) == (unsigned)T - 1u) {
      __threadfence();
      const uint32_t total_out = atomicExch(&cacc->x, 0u);
      atomicExch(&cacc->y, 0u);
      if (checked && s_code == EBC_OK && fail == EBC_OK && !dec_aborted(g, epoch) &&
          (unsigned long long)total_out != L.n_out)
        dec_fail(g, epoch, EBC_ERR_CORRUPT);
    }
  }
}

// ---------------------------------------------------------------------------
// k_dec_match: persistent warps over the bitmap words of all units (32 rows
// each): every matched row of the word copies its reference row -- the literal
// the reference names (whole batch; checked to precede the row and to be a
// literal), or the literal root of its chain (window; resolved by k_dec_lit).
// A lane copies 16 bytes of a row, kUnroll rows' worth in flight.
// ---------------------------------------------------------------------------
constexpr int kMatchThreads = 256;
struct MLay {                    // what the match copy needs of a container
  unsigned long long base, off_bm, off_refs, off_seg, row0;
  unsigned int n, nseg, nw, ref_bytes, window;
};
template <int D>
__global__ void __launch_bounds__(kMatchThreads, 4) k_dec_match(const uint8_t* __restrict__ in,
                                                               unsigned long long in_bytes,
                                                               const unsigned long long* __restrict__ offs, Shape sh,
                                                               Work w, float* __restrict__ xhat, uint32_t epoch) {
  pdl_enter();
  using G = DGeo<D>;
  constexpr int kQ = D / 4;                         // float4 per row
  constexpr int kUnroll = 4;                        // float4 per lane in flight
  constexpr int kNW = kMatchThreads / 32;
  __shared__ MLay s_lay[kMaxSlices];
  __shared__ uint32_t s_dst[kNW][32], s_src[kNW][32];
  __shared__ int s_abort;
  Glob* g = w.glob;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) s_abort = dec_aborted(g, epoch);
  __syncthreads();
  if (s_abort) return;
  for (int c = tid; c < sh.R; c += kMatchThreads) {   // the containers' layouts, as k_dec_lit checked them
    const Layout Lc = w.lay[c];
    s_lay[c] = MLay{Lc.base, Lc.off_bitmap, Lc.off_refs, Lc.off_seg, Lc.row0, (unsigned int)Lc.n, Lc.nseg, Lc.nw,
                    Lc.ref_bytes, Lc.window};
  }
  __syncthreads();
  const int T = sh.T;
  const unsigned long long nbatch = (unsigned long long)sh.U * sh.nw;   // bitmap words of all units
  const unsigned long long wstep = (unsigned long long)gridDim.x * kNW;
  for (unsigned long long k = (unsigned long long)blockIdx.x * kNW + warp; k < nbatch; k += wstep) {
    // words go unit-fastest: the rows written at a time are whole rows of the output
    const unsigned int wi = (unsigned int)(k / (unsigned long long)sh.U);
    const int u = (int)(k - (unsigned long long)wi * sh.U);
    const int r = u / T, t = u - r * T;
    const MLay& Lc = s_lay[r];
    if (wi >= Lc.nw) continue;
    const uint8_t* cin = in + Lc.base;
    const uint32_t* bmt = reinterpret_cast<const uint32_t*>(cin + Lc.off_bm) + (size_t)t * Lc.nw;
    const uint32_t bm = bmt[wi];
    if (bm == 0u) continue;
    // the rank of the word's first match: the segment's match base + the matches of its earlier words
    const unsigned int s = wi / G::kBmWords, wfirst = s * G::kBmWords;
    uint32_t before = 0;
    for (unsigned int i = wfirst + lane; i < wi; i += 32) before += __popc(bmt[i]);
    before = __reduce_add_sync(0xffffffffu, before);
    const uint32_t mbase =
        reinterpret_cast<const uint32_t*>(cin + Lc.off_seg)[4ull * ((unsigned long long)t * Lc.nseg + s) + 2];
    const int64_t b = (int64_t)wi * 32 + lane;   // row of the slice
    const bool m = (bm >> lane) & 1u;
    const uint32_t at = __popc(bm & ((1u << lane) - 1u));
    bool good = true;
    if (m) {
      uint32_t ref;
      if (Lc.window) {   // the chain's literal root, resolved by k_dec_lit
        ref = __ldcg(&w.srcrow[(size_t)t * sh.B + Lc.row0 + b]) - (uint32_t)Lc.row0;
        good = ref < (uint32_t)b;
      } else {           // whole slice: the first occurrence, always a literal
        const unsigned long long kk = (unsigned long long)mbase + before + at;
        const uint8_t* refs = cin + Lc.off_refs;
        ref = Lc.ref_bytes == 2 ? (uint32_t)reinterpret_cast<const uint16_t*>(refs)[kk]
                                : reinterpret_cast<const uint32_t*>(refs)[kk];
        good = (int64_t)ref < b && !((bmt[ref >> 5] >> (ref & 31)) & 1u);
      }
      s_dst[warp][at] = (uint32_t)b;
      s_src[warp][at] = good ? ref : (uint32_t)b;
    }
    if (!__all_sync(0xffffffffu, good)) {
      if (lane == 0) dec_fail(g, epoch, EBC_ERR_CORRUPT);
      return;
    }
    __syncwarp();
    const uint32_t nm = __popc(bm);
    const size_t rstride = (size_t)sh.T_out * D;   // floats between consecutive batch rows
    float* base = xhat + ((size_t)Lc.row0 * sh.T_out + sh.t_off + t) * D;
    // (row, float4) pairs of the word's matched rows, kUnroll per lane in flight
    for (uint32_t p0 = 0; p0 < nm * kQ; p0 += 32u * kUnroll) {
      float4 v[kUnroll];
      float4* dp[kUnroll];
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const uint32_t pi = p0 + (uint32_t)i * 32u + lane;
        dp[i] = nullptr;
        if (pi < nm * kQ) {
          const uint32_t row = pi / kQ, q = pi % kQ;
          v[i] = __ldcg(reinterpret_cast<const float4*>(base + (size_t)s_src[warp][row] * rstride) + q);
          dp[i] = reinterpret_cast<float4*>(base + (size_t)s_dst[warp][row] * rstride) + q;
        }
      }
#pragma unroll
      for (int i = 0; i < kUnroll; ++i)
        if (dp[i]) __stcs(dp[i], v[i]);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D, int W>
static void launch_decompress_d(const uint8_t* in, unsigned long long in_bytes, const unsigned long long* offs,
                                const Shape& sh, const Work& w, float* xhat, uint32_t epoch, cudaStream_t st,
                                Prof* prof) {
  using G = DGeo<D>;
  const unsigned ngrp = (unsigned)(div_up(sh.nseg, G::kSPC) > 0 ? div_up(sh.nseg, G::kSPC) : 1);
  unsigned nshare = ngrp;
  if (G::kKC == 1 && sh.nseg > 0 && sh.nseg <= kDecShareMaxSeg && sh.U > 0) {
    // decode shares: as many CTAs per unit as are resident at once (at least one per group)
    static int per_sm = -1;
    if (per_sm < 0 && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dec_lit<D, W>, G::kThreads, 0) !=
                           cudaSuccess ||
                       per_sm < 1))
      per_sm = 1;
    const unsigned fit = (unsigned)((sh.nsm > 0 ? sh.nsm : 152) * per_sm) / (unsigned)sh.U;
    if (fit > nshare) nshare = fit;   // (else the groups decode their own chunks)
  }
  const unsigned grid = sh.U > 0 ? (unsigned)sh.U * nshare : 1u;
  prof_begin(prof, "k_dec_lit", st);
  launch_k(k_dec_lit<D, W>, grid, G::kThreads, 0, st, in, in_bytes, offs, sh, w, xhat, epoch, (int)nshare);
  prof_end(prof, st);
  if (sh.U > 0 && sh.nseg > 0) {
    // persistent: the resident CTAs, at most one warp per bitmap word
    const unsigned long long words = (unsigned long long)sh.U * sh.nw;
    unsigned mgrid = (unsigned)((sh.nsm > 0 ? sh.nsm : 152) * 4);
    const unsigned long long need = (words + kMatchThreads / 32 - 1) / (kMatchThreads / 32);
    if (need < mgrid) mgrid = (unsigned)need;
    prof_begin(prof, "k_dec_match", st);
    launch_k(k_dec_match<D>, mgrid, kMatchThreads, 0, st, in, in_bytes, offs, sh, w, xhat, epoch);
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

cudaError_t set_decoder_attributes() { return cudaSuccess; }   // every decoder kernel fits the default limits

}  // namespace ebc
