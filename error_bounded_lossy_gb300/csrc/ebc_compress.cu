// ebc_compress.cu -- compression kernels of the error-bounded embedding codec.
//
// Method: "Accelerating Communication in Deep Learning Recommendation Model
// Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
// §III-D (quantization encoder, vector-based LZ, Huffman) and §III-E (one
// output buffer, chunk offsets found on the device; with "Buffer
// Optimization", one container per batch slice in the same pass).  The coding
// unit is a table of one slice (a table when there is one slice).  Up to five
// launches on the caller's stream:
//   k_quantize  x -> codes and per-vector dedup keys (TMA-staged input tiles);
//               then the keys of its rows -> per-unit first-occurrence hash tables
//   k_resolve   literal / match decision; literal code histograms per segment
//               and per unit
//   k_codebook  per-unit Huffman code (and, for units of at most 256 segments,
//               their segment offsets); the last CTA lays out the containers
//               and writes the headers
//   k_layout    (units of more than 256 segments) per segment bit counts and
//               offsets; its last CTA completes the containers
//   k_emit      per segment: bitstream, chunk index, references, records;
//               empties its share of the hash tables
// All offsets come from prefix sums, never from atomic reservations, so the
// container is byte-identical from run to run.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <type_traits>

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
// Four codes packed into one word (code of element k in byte k), branch-free:
// for an accepted q the low byte of y's bits is q mod 256, so code = byte ^ 0x80;
// a rejected element takes the byte 0x80, which becomes code 0.
__device__ __forceinline__ uint32_t quantize_four(float4 v, float eb, float ebx2, float inv, bool ok[4]) {
  const float xs[4] = {v.x, v.y, v.z, v.w};
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float t = __fmul_rn(xs[k], inv);
    const float y = __fadd_rn(t, 12582912.0f);       // 1.5 * 2^23
    const float qf = __fsub_rn(y, 12582912.0f);      // exact when |t| < 2^22
    const float err = fabsf(__fsub_rn(xs[k], __fmul_rn(qf, ebx2)));
    ok[k] = (fabsf(t) < 127.5f) & (err <= eb);        // false for NaN and +-inf too
    u[k] = ok[k] ? __float_as_uint(y) : 0x80u;
  }
  return __byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u) ^ 0x80808080u;
}

// The wide alphabet (radius 512): four 16-bit codes q + 512 in two words.  The
// low half-word of y's bits is q mod 2^16; a rejected element takes 0xFE00,
// and a per-half-word add of 512 (no carry between the halves) gives the code.
__device__ __forceinline__ uint2 quantize_four_wide(float4 v, float eb, float ebx2, float inv, bool ok[4]) {
  const float xs[4] = {v.x, v.y, v.z, v.w};
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float t = __fmul_rn(xs[k], inv);
    const float y = __fadd_rn(t, 12582912.0f);       // 1.5 * 2^23
    const float qf = __fsub_rn(y, 12582912.0f);      // exact when |t| < 2^22
    const float err = fabsf(__fsub_rn(xs[k], __fmul_rn(qf, ebx2)));
    ok[k] = (fabsf(t) < 511.5f) & (err <= eb);        // false for NaN and +-inf too
    u[k] = ok[k] ? __float_as_uint(y) : 0xFE00u;
  }
  return make_uint2(__vadd2(__byte_perm(u[0], u[1], 0x5410u), 0x02000200u),
                    __vadd2(__byte_perm(u[2], u[3], 0x5410u), 0x02000200u));
}

template <int W>
__device__ __forceinline__ typename QuadOf<W>::T quantize_quad(float4 v, float eb, float ebx2, float inv, bool ok[4]) {
  if constexpr (W == 1) return quantize_four(v, eb, ebx2, inv, ok);
  else return quantize_four_wide(v, eb, ebx2, inv, ok);
}

// The same arithmetic on pairs of values with the packed (two-lane) fp32
// instructions: t = fl(x * inv), y = fl(t + 1.5*2^23), q = fl(y - 1.5*2^23),
// h = fl(q * ebx2), each rounded to nearest as in the scalar form.  The error
// x - h is taken with the scalar, explicitly rounded subtraction: a packed
// subtraction after the packed product is contracted into one fused
// multiply-add by the compiler (even written as an fma with a -0 addend),
// which rounds x - q * ebx2 once and moves the error bound's edge.
// inv2, ebx22, c2: the operands duplicated in both halves.
__device__ __forceinline__ void quantize_pair(float x0, float x1, unsigned long long inv2, unsigned long long ebx22,
                                              unsigned long long c2, float& t0, float& t1, float& y0, float& y1,
                                              float& e0, float& e1) {
  float h0, h1;
  asm("{\n .reg .b64 X, T, Y, Q, H;\n"
      " mov.b64 X, {%6, %7};\n"
      " mul.rn.f32x2 T, X, %8;\n"
      " add.rn.f32x2 Y, T, %10;\n"
      " sub.rn.f32x2 Q, Y, %10;\n"
      " mul.rn.f32x2 H, Q, %9;\n"
      " mov.b64 {%0, %1}, T;\n mov.b64 {%2, %3}, Y;\n mov.b64 {%4, %5}, H;\n}"
      : "=f"(t0), "=f"(t1), "=f"(y0), "=f"(y1), "=f"(h0), "=f"(h1)
      : "f"(x0), "f"(x1), "l"(inv2), "l"(ebx22), "l"(c2));
  e0 = __fsub_rn(x0, h0);
  e1 = __fsub_rn(x1, h1);
}
__device__ __forceinline__ unsigned long long dup2(float v) {
  return ((unsigned long long)__float_as_uint(v) << 32) | __float_as_uint(v);
}

// Four codes from the packed quantizer: ok[k] when |t| < R - 1/2 and |err| <= eb.
template <int W>
__device__ __forceinline__ typename QuadOf<W>::T quantize_quad2(float4 v, float eb, unsigned long long inv2,
                                                                unsigned long long ebx22, bool ok[4]) {
  constexpr float kLim = W == 1 ? 127.5f : 511.5f;
  const unsigned long long c2 = 0x4B4000004B400000ull;   // 1.5 * 2^23 in both halves
  float t[4], y[4], e[4];
  quantize_pair(v.x, v.y, inv2, ebx22, c2, t[0], t[1], y[0], y[1], e[0], e[1]);
  quantize_pair(v.z, v.w, inv2, ebx22, c2, t[2], t[3], y[2], y[3], e[2], e[3]);
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ok[k] = (fabsf(t[k]) < kLim) & (fabsf(e[k]) <= eb);   // false for NaN and +-inf too
    u[k] = ok[k] ? __float_as_uint(y[k]) : (W == 1 ? 0x80u : 0xFE00u);
  }
  if constexpr (W == 1) {
    return __byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u) ^ 0x80808080u;
  } else {
    return make_uint2(__vadd2(__byte_perm(u[0], u[1], 0x5410u), 0x02000200u),
                      __vadd2(__byte_perm(u[2], u[3], 0x5410u), 0x02000200u));
  }
}

// The dedup key's terms for four codes at element d of the row: one word of
// four codes, or two words of two codes (word index k = d / 4 or d / 2).
__device__ __forceinline__ uint32_t quad_key(uint32_t v, int d) {
  return lowbias32(v + (uint32_t)(d >> 2) * 0x9E3779B9u);
}
__device__ __forceinline__ uint32_t quad_key(uint2 v, int d) {
  return lowbias32(v.x + (uint32_t)(d >> 1) * 0x9E3779B9u) + lowbias32(v.y + (uint32_t)((d >> 1) + 1) * 0x9E3779B9u);
}

// Four codes from the code scratch (element index e of a table; W bytes each).
__device__ __forceinline__ uint32_t ld_quad(const uint8_t* symt, size_t e, uint32_t*) {
  return __ldcg(reinterpret_cast<const unsigned int*>(symt + e));
}
__device__ __forceinline__ uint2 ld_quad(const uint8_t* symt, size_t e, uint2*) {
  return __ldcg(reinterpret_cast<const uint2*>(symt + 2 * e));
}
// ... and from a shared-memory copy, at 32-bit word index i (even for W = 2)
__device__ __forceinline__ uint32_t sm_quad(const uint32_t* s, int i, uint32_t*) { return s[i]; }
__device__ __forceinline__ uint2 sm_quad(const uint32_t* s, int i, uint2*) {
  return *reinterpret_cast<const uint2*>(s + i);
}
// Code c of 16 bytes of codes (W bytes each), and whether one of them is 0.
template <int W>
__device__ __forceinline__ uint32_t v4_code(const uint4& v, int c) {
  constexpr int kPerWord = 4 / W;
  const int k = c / kPerWord;
  const uint32_t x = k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
  return (x >> (8 * W * (c % kPerWord))) & (W == 1 ? 0xffu : 0xffffu);
}
template <int W>
__device__ __forceinline__ bool v4_has_zero(const uint4& v) {
  if constexpr (W == 1)
    return quad_has_zero(v.x) || quad_has_zero(v.y) || quad_has_zero(v.z) || quad_has_zero(v.w);
  else
    return quad_has_zero(make_uint2(v.x, v.y)) || quad_has_zero(make_uint2(v.z, v.w));
}
__device__ __forceinline__ bool v4_eq(const uint4& a, const uint4& b) {
  return ((a.x ^ b.x) | (a.y ^ b.y) | (a.z ^ b.z) | (a.w ^ b.w)) == 0u;
}

// Input element types: fp32, or bf16 carried as its 16 raw bits (its fp32
// value is exact: the bf16 bits followed by 16 zero bits).
__device__ __forceinline__ uint32_t raw32(float v) { return __float_as_uint(v); }
__device__ __forceinline__ uint32_t raw32(uint16_t v) { return (uint32_t)v << 16; }
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const uint16_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ unsigned long long l2_evict_last() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Code scratch is written once and read twice more; keep it in L2 while the
// read-once input streams through.
__device__ __forceinline__ void st_keep_u32(uint32_t* p, uint32_t v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
// Four codes into the code scratch at element e of a table.
__device__ __forceinline__ void st_keep_quad(uint8_t* symt, size_t e, uint32_t v, unsigned long long pol) {
  st_keep_u32(reinterpret_cast<uint32_t*>(symt + e), v, pol);
}
__device__ __forceinline__ void st_keep_quad(uint8_t* symt, size_t e, uint2 v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;" ::"l"(symt + 2 * e), "r"(v.x), "r"(v.y), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void dedup_insert(unsigned long long* slots, uint32_t S, uint32_t h, uint32_t b,
                                             Glob* g) {
  // First occurrence per key: the slot keeps (h << 32 | min row); keys that
  // collide on the slot index probe linearly.  A slot already holding the key
  // needs no returning atomic.
  const unsigned long long mine = ((unsigned long long)h << 32) | b;
  uint32_t slot = h & (S - 1);
  for (uint32_t p = 0; p < S; ++p) {
    unsigned long long cur = __ldcg(slots + slot);
    if (cur == kEmptySlot) {
      cur = atomicCAS(slots + slot, kEmptySlot, mine);
      if (cur == kEmptySlot) return;
    }
    if ((uint32_t)(cur >> 32) == h) {
      if (cur > mine) atomicMin(slots + slot, mine);
      return;
    }
    slot = (slot + 1) & (S - 1);
  }
  record_error(g, EBC_ERR_INTERNAL);
}

__device__ __forceinline__ uint32_t dedup_lookup(const unsigned long long* slots, uint32_t S, uint32_t h,
                                                 Glob* g) {
  uint32_t slot = h & (S - 1);
  for (uint32_t p = 0; p < S; ++p) {
    const unsigned long long v = __ldcg(slots + slot);
    if (v == kEmptySlot) break;
    if ((uint32_t)(v >> 32) == h) return (uint32_t)v;
    slot = (slot + 1) & (S - 1);
  }
  record_error(g, EBC_ERR_INTERNAL);
  return 0xFFFFFFFFu;
}

// ---------------------------------------------------------------------------
// Tensor-memory-accelerator (TMA) staging of input tiles.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte asynchronous global -> shared copies (completion by commit/wait groups)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Bounded wait for phase `parity` of an mbarrier (at most `limit` polls); false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit = kWaitLimit) {
  for (int i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// The input is read once: its lines are the first the L2 gives up (policy from
// createpolicy), so the code scratch written meanwhile stays resident for the
// kernels that read it again.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Box geometry of one segment's input tile x[row0 .. row0+SB)[t][0 .. D):
// boxes of at most 256 rows x 256 elements; box (rb, db) lands at
// ((rb * kNBoxD + db) * kBoxR) * kBoxD floats in the stage.
template <int D, typename In = float>
struct QGeo {
  static constexpr int kBoxD = D < 256 ? D : 256;
  static constexpr int kBoxR = Geo<D>::kSB < 256 ? Geo<D>::kSB : 256;
  static constexpr int kNBoxD = D / kBoxD;
  static constexpr int kNBoxR = Geo<D>::kSB / kBoxR;
  static constexpr int kStageFloats = Geo<D>::kSegSyms;
  static constexpr uint32_t kStageBytes = (uint32_t)kStageFloats * (uint32_t)sizeof(In);
  __device__ static __forceinline__ int offset(int r, int d) {
    return (((r / kBoxR) * kNBoxD + d / kBoxD) * kBoxR + r % kBoxR) * kBoxD + d % kBoxD;
  }
};

template <int D, typename In>
__device__ __forceinline__ void issue_segment_tile(In* stage, const CUtensorMap* map, uint64_t* bar, const Shape& sh,
                                                   int seg) {
  using Q = QGeo<D, In>;
  const int s = seg / sh.T;   // segments go table-fastest: tiles in flight cover whole rows
  const int t = seg - s * sh.T;
  unsigned long long first;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(first));
  mbar_expect_tx(bar, Q::kStageBytes);
#pragma unroll
  for (int rb = 0; rb < Q::kNBoxR; ++rb)
#pragma unroll
    for (int db = 0; db < Q::kNBoxD; ++db)
      tma_load_3d(stage + ((rb * Q::kNBoxD + db) * Q::kBoxR) * Q::kBoxD, map, bar, db * Q::kBoxD, t,
                  s * Geo<D>::kSB + rb * Q::kBoxR, first);
}

// ---------------------------------------------------------------------------
// k_quantize: persistent CTAs, each taking segments blockIdx.x, +gridDim.x, ...
// A segment's input tile (rows of one table) arrives in shared memory by TMA
// into one of two stages, so the next tile streams in while the current one is
// quantized.  After its last tile the CTA enters the keys of all its rows into
// the first-occurrence tables (lanes holding the same key are merged with
// match.any first, so hot keys queue fewer atomics); other CTAs are still
// streaming meanwhile.  8 warps, each a run of 128-element
// slabs (lane = 4 consecutive elements).  The dedup key of a vector is the
// wrapping sum over its 4-code words w_k of lowbias32(w_k + k * 0x9E3779B9)
// plus lowbias32(raw ^ (d + 1) * 0x85EBCA6B) for each outlier at position d.
// ---------------------------------------------------------------------------
template <int D, typename In, int W>
__global__ void __launch_bounds__(256) k_quantize(const __grid_constant__ CUtensorMap tmap, Shape sh, EbParams ep,
                                                   Work w, uint32_t epoch) {
  pdl_enter();
  using G = Geo<D>;
  using Q = QGeo<D, In>;
  using Quad = typename QuadOf<W>::T;
  constexpr int kA = Alph<W>::kA;
  extern __shared__ __align__(128) unsigned char s_raw[];   // 2 stages of kStageFloats elements, then T x {2 eb, 1/(2 eb)}
  In* s_x = reinterpret_cast<In*>(s_raw);
  float2* s_tab = reinterpret_cast<float2*>(s_raw + 2 * Q::kStageBytes);
  __shared__ __align__(8) uint64_t s_bar[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsegT = sh.T * sh.qseg;
  const int64_t B = sh.B;
  const unsigned long long pol = l2_evict_last();
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if ((int)blockIdx.x < nsegT) issue_segment_tile<D, In>(s_x, &tmap, &s_bar[0], sh, blockIdx.x);
    if ((int)(blockIdx.x + gridDim.x) < nsegT)
      issue_segment_tile<D, In>(s_x + Q::kStageFloats, &tmap, &s_bar[1], sh, blockIdx.x + gridDim.x);
  }
  for (int t = tid; t < sh.T; t += 256) {   // each table's 2 eb and its reciprocal, once per CTA
    const float ebx2 = __fmul_rn(2.0f, ep.eb[t]);
    s_tab[t] = make_float2(ebx2, __fdiv_rn(1.0f, ebx2));
  }
  __syncthreads();
  uint32_t parity = 0;   // bit i: phase of stage i
  int i = 0;
  for (int seg = blockIdx.x; seg < nsegT; seg += gridDim.x, ++i) {
    const int stg = i & 1;
    const In* xs = s_x + stg * Q::kStageFloats;
    const int s = seg / sh.T;
    const int t = seg - s * sh.T;
    const int64_t row0 = (int64_t)s * G::kSB;
    if (s == 0) {   // per-call accumulators of the table's units, which k_resolve adds to
      for (int r = 0; r < sh.R; ++r) {
        const int u = r * sh.T + t;
        for (int k = tid; k < kA; k += 256) w.tab_hist[(size_t)u * kA + k] = 0u;
        if (tid == 0) w.tab_cnt[u] = make_uint4(0, 0, 0, 0);
      }
    }
    const float eb = ep.eb[t];
    const float2 tb = s_tab[t];
    const unsigned long long ebx22 = dup2(tb.x), inv2 = dup2(tb.y);
    const int nrows = (int)min((int64_t)G::kSB, B - row0);          // rows of the segment in the batch
    uint8_t* symseg = w.sym + (size_t)t * sh.symstride + (size_t)row0 * D * W;
    uint32_t* hseg = w.vhash + (size_t)t * B + row0;
    const bool arrived = mbar_wait(&s_bar[stg], (parity >> stg) & 1u, i == 0 ? sh.first_wait : kWaitLimit);
    if (__syncthreads_or(!arrived)) {   // the whole CTA stops together
      if (tid == 0) {
        record_error(w.glob, EBC_ERR_DEVICE_TIMEOUT);
        // the call is given up: the kernels after this one write nothing to the output
        atomicExch(&w.glob->cabort, status_word(epoch, EBC_ERR_DEVICE_TIMEOUT));
        // no copy may still be writing into this CTA's shared memory when it exits: wait (with
        // the full limit) for this stage's tile and for the next one, if it was issued
        if (!arrived) mbar_wait(&s_bar[stg], (parity >> stg) & 1u);
        if (seg + (int)gridDim.x < nsegT) mbar_wait(&s_bar[stg ^ 1], (parity >> (stg ^ 1)) & 1u);
      }
      __syncthreads();
      return;
    }
    parity ^= 1u << stg;
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < G::kSlabsPerWarp; ++k) {
      const int slab = warp * G::kSlabsPerWarp + k;
      const int e = slab * 128 + lane * 4;   // element of the segment
      const int r = e / D;                   // row of the segment
      const int d = e % D;
      const bool valid = r < nrows;
      const float4 v = load4(xs + Q::offset(r, d));
      bool ok[4];
      const Quad word = quantize_quad2<W>(v, eb, inv2, ebx22, ok);
      if (valid) st_keep_quad(symseg, (size_t)e, word, pol);
      acc += quad_key(word, d);
      if (!(ok[0] & ok[1] & ok[2] & ok[3])) {
        if (!ok[0]) acc += lowbias32(raw32(xs[Q::offset(r, d) + 0]) ^ (uint32_t)(d + 1) * 0x85EBCA6Bu);
        if (!ok[1]) acc += lowbias32(raw32(xs[Q::offset(r, d) + 1]) ^ (uint32_t)(d + 2) * 0x85EBCA6Bu);
        if (!ok[2]) acc += lowbias32(raw32(xs[Q::offset(r, d) + 2]) ^ (uint32_t)(d + 3) * 0x85EBCA6Bu);
        if (!ok[3]) acc += lowbias32(raw32(xs[Q::offset(r, d) + 3]) ^ (uint32_t)(d + 4) * 0x85EBCA6Bu);
      }
      if ((slab + 1) % G::kSPR == 0) {            // the row ends with this slab: its key, over its kLPR lanes
        if constexpr (G::kLPR == 32) {
          acc = __reduce_add_sync(0xffffffffu, acc);
        } else {
#pragma unroll
          for (int off = G::kLPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        }
        if (valid && (lane % G::kLPR) == 0) hseg[r] = acc;
        acc = 0;
      }
    }
    __syncthreads();   // the stage is consumed: refill it with the segment two steps ahead
    if (tid == 0 && seg + 2 * (int)gridDim.x < nsegT)
      issue_segment_tile<D, In>(s_x + stg * Q::kStageFloats, &tmap, &s_bar[stg], sh, seg + 2 * gridDim.x);
  }
  if (sh.window == 0 && (int)blockIdx.x < nsegT) {
    // the keys of this CTA's rows into the first-occurrence tables, after its last tile
    __syncthreads();
    const int nmine = (nsegT - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int total = nmine * G::kSB;   // a multiple of 32: a warp's rows lie in one segment
    for (int i = tid; i < total; i += 256) {
      const int seg = (int)blockIdx.x + (i / G::kSB) * (int)gridDim.x;
      const int st = seg / sh.T;
      const int t = seg - st * sh.T;
      const int64_t b = (int64_t)st * G::kSB + i % G::kSB;
      const bool valid = b < B && !(table_mode(w, t) & kModeNoDedup);
      // each slice keeps its own table: a row never refers into another slice
      const int u = valid ? slice_of_row(sh, b) * sh.T + t : 0;
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t h = __ldcg(&w.vhash[(size_t)t * B + b]);
        const unsigned same = sh.R == 1 ? __match_any_sync(vmask, h)
                                        : __match_any_sync(vmask, ((unsigned long long)u << 32) | h);
        if (lane == __ffs(same) - 1) dedup_insert(w.slots + (size_t)u * sh.S, sh.S, h, (uint32_t)b, w.glob);
      }
    }
  }
}


// ---------------------------------------------------------------------------
// k_resolve: vector-based LZ with the whole batch as window and the first
// occurrence as reference (§III-D, §III-E "fixed pattern length"): row b is a
// match when the first row with its key precedes it and carries the same codes
// and the same raw bits at outliers; otherwise a literal (a key collision is a
// literal too).  Literal codes feed the segment and table histograms.  Rows
// of 16 bytes or more are compared 16 bytes per lane (a warp step covers
// 32 * 16 bytes of rows), and the literal rows are listed; their codes then go
// into the warp's histogram in a second pass.  Shorter rows are compared and
// counted in one pass, four codes per lane.
// ---------------------------------------------------------------------------
constexpr int kResolveThreads = 64;   // two warps per segment: many segments in flight per SM

template <int D, typename In, int W>
__global__ void __launch_bounds__(kResolveThreads) k_resolve(const In* __restrict__ x, Shape sh, Work w) {
  pdl_enter();
  using G = Geo<D>;
  using Quad = typename QuadOf<W>::T;
  constexpr int kA = Alph<W>::kA;
  constexpr int kNT = kResolveThreads, kNW = kNT / 32;
  constexpr int kRPT = (G::kSB + kNT - 1) / kNT;          // rows per thread in the lookups
  constexpr int kSteps = G::kSB / kNW / G::kRPS;         // warp steps (kRPS rows each) per warp
  constexpr int kGroup = kSteps < 8 ? kSteps : 8;        // steps whose loads are issued together
  // window mode: keys of rows row0 - window .. row0 + SB during the lookups; then the literal
  // code histograms, one per warp
  constexpr int kHistWin = kNW * kA > kMaxWindow + G::kSB ? kNW * kA : kMaxWindow + G::kSB;
  __shared__ __align__(16) uint32_t s_histwin[kHistWin];
  uint32_t* s_win = s_histwin;
  __shared__ __align__(16) uint32_t s_sym[G::kSegSyms * W / 4 + 4];   // the segment's own codes
  __shared__ uint32_t s_ref[G::kSB];
  __shared__ uint32_t s_bm[G::kBmWords];
  __shared__ uint32_t s_cnt[3];
  // rows of 16 bytes or more: the match test takes 16 bytes of codes per lane
  constexpr bool kWide = D * W >= 16;
  constexpr int kRU = kWide ? D * W / 16 : 1;          // 16-byte pieces of a row
  constexpr int kLPV = kRU < 32 ? kRU : 32;            // lanes per row
  constexpr int kUPL = kRU / kLPV;                     // pieces per lane
  constexpr int kRPV = 32 / kLPV;                      // rows per warp step
  constexpr int kStepsV = G::kSB / kNW / kRPV;         // warp steps per warp
  constexpr int kGV = kStepsV < 4 ? kStepsV : 4;       // steps whose loads are issued together
  __shared__ uint16_t s_lit[kWide ? G::kSB : 1];       // each warp's literal rows, in its half
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < G::kBmWords; i += kNT) s_bm[i] = 0u;
  if (tid < 3) s_cnt[tid] = 0u;

  // segment s of unit u = (slice r, table t): rows b0 + s * SB .. of the batch
  const int seg = blockIdx.x;
  const int u = seg / sh.nseg;
  const int s = seg - u * sh.nseg;
  const int r = u / sh.T;
  const int t = u - r * sh.T;
  const int64_t B = sh.B;
  const int T = sh.T;
  const int64_t b0 = slice_row0(sh, r);
  const int64_t bend = b0 + slice_rows(sh, r);              // rows of the slice: [b0, bend)
  const int64_t row0 = b0 + (int64_t)s * G::kSB;
  const unsigned long long* slots = w.slots + (size_t)u * sh.S;
  const uint8_t* symt = w.sym + (size_t)t * sh.symstride;
  const bool nodedup = (table_mode(w, t) & kModeNoDedup) != 0;   // every row its own reference
  // the segment's codes start so words into s_sym (a slice may start off a 16-byte boundary when
  // D * W < 16; so is even when W = 2)
  const int so = D * W >= 16 ? 0 : (int)(((size_t)row0 * D * W) & 15u) / 4;
  {   // the segment's codes (rows contiguous; the table stride is padded to 16 bytes), copied
      // asynchronously while the keys are looked up
    const int64_t nrows = bend - row0 < G::kSB ? bend - row0 : G::kSB;
    const int nq = nrows > 0 ? (int)((so * 4 + nrows * D * W + 15) / 16) : 0;
    const uint4* src = reinterpret_cast<const uint4*>(symt + (size_t)row0 * D * W - so * 4);
    for (int i = tid; i < nq; i += kNT) cp_async16(reinterpret_cast<uint4*>(s_sym) + i, src + i);
  }
  if (sh.window > 0 && !nodedup) {
    // window: the nearest earlier row of the slice within the window with the same key
    // (the keys of the window and the segment, in shared memory)
    const int64_t lo = row0 - sh.window > b0 ? row0 - sh.window : b0;
    const int64_t hi = row0 + G::kSB < bend ? row0 + G::kSB : bend;
    for (int64_t i = tid; i < hi - lo; i += kNT) s_win[i] = __ldcg(&w.vhash[(size_t)t * B + lo + i]);
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < kRPT; ++k) {
      const int rr = k * kNT + tid;
      const int64_t b = row0 + rr;
      if (rr < G::kSB && b < bend) {
        const uint32_t h = s_win[b - lo];
        const int64_t stop = b - sh.window > lo ? b - sh.window : lo;
        uint32_t ref = (uint32_t)b;
        for (int64_t c2 = b - 1; c2 >= stop; --c2)
          if (s_win[c2 - lo] == h) {
            ref = (uint32_t)c2;
            break;
          }
        s_ref[rr] = ref;
      }
    }
  } else
  // one thread per row: first occurrence of the row's key in the slice
  {
    uint32_t h[kRPT];
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const int rr = k * kNT + tid;
      const int64_t b = row0 + rr;
      if (rr < G::kSB && b < bend) h[k] = __ldcg(&w.vhash[(size_t)t * B + b]);
    }
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const int rr = k * kNT + tid;
      const int64_t b = row0 + rr;
      if (rr < G::kSB && b < bend) {
        uint32_t ref = nodedup ? (uint32_t)b : dedup_lookup(slots, sh.S, h[k], w.glob);
        if (ref > (uint32_t)b || (int64_t)ref < b0) ref = (uint32_t)b;   // only on an internal error
        s_ref[rr] = ref;
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  for (int i = tid; i < kNW * kA / 4; i += kNT)   // the window keys are no longer needed
    reinterpret_cast<uint4*>(s_histwin)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  uint32_t* hist = s_histwin + warp * kA;
  uint32_t n_lit = 0, n_match = 0;
  if constexpr (kWide) {
    // ---- rows of at least 16 bytes: first the match test, 16 bytes of codes per lane (kLPV lanes
    //      per row, kRPV rows per warp step), with the reference rows of kGV steps in flight ----
    const int sub = lane % kLPV;   // the lane's 16 bytes of its row: sub + k * kLPV, k < kUPL
    const unsigned gmask = (kLPV == 32 ? 0xffffffffu : ((1u << kLPV) - 1u)) << (lane & ~(kLPV - 1));
    const bool leader = sub == 0;
    const unsigned below = (1u << lane) - 1u;
    uint16_t* lits = s_lit + warp * (G::kSB / kNW);   // this warp's literal rows (row of the segment)
    int nlw = 0;                                      // ... and their number (the same in every lane)
    auto load_refs = [&](int g0, uint4 (&rv)[kGV][kUPL]) {
#pragma unroll
      for (int it = 0; it < kGV; ++it) {
        const int rr = (warp * kStepsV + g0 + it) * kRPV + lane / kLPV;
        const int64_t b = row0 + rr;
        const uint32_t ref = b < bend ? s_ref[rr] : (uint32_t)b;
        const uint4* rp = reinterpret_cast<const uint4*>(symt + (size_t)ref * (D * W)) + sub;
#pragma unroll
        for (int k = 0; k < kUPL; ++k) rv[it][k] = ref != (uint32_t)b ? __ldcg(rp + k * kLPV) : make_uint4(0, 0, 0, 0);
      }
    };
    auto test = [&](int g0, const uint4 (&rv)[kGV][kUPL]) {
#pragma unroll
      for (int it = 0; it < kGV; ++it) {
        const int rr = (warp * kStepsV + g0 + it) * kRPV + lane / kLPV;
        const int64_t b = row0 + rr;
        const bool valid = b < bend;
        const uint32_t ref = valid ? s_ref[rr] : 0u;
        const bool cand = valid && ref != (uint32_t)b;
        bool eq = true;
#pragma unroll
        for (int k = 0; k < kUPL; ++k) {
          const uint4 ov = reinterpret_cast<const uint4*>(s_sym)[rr * (D * W / 16) + sub + k * kLPV];
          bool e = v4_eq(ov, rv[it][k]);
          if (cand && e && v4_has_zero<W>(ov)) {   // outliers: their raw bits must agree too
            const int d0 = (sub + k * kLPV) * (16 / W);
            const In* xb = x + ((size_t)b * T + t) * D + d0;
            const In* xr = x + ((size_t)ref * T + t) * D + d0;
            for (int c = 0; c < 16 / W; ++c)
              if (v4_code<W>(ov, c) == 0u && raw32(xb[c]) != raw32(xr[c])) e = false;
          }
          eq = eq && e;
        }
        const unsigned bad = __ballot_sync(0xffffffffu, !eq);
        const bool match = cand && (bad & gmask) == 0u;
        if (valid && leader && match) {
          w.ref[(size_t)t * B + b] = ref;
          atomicOr(&s_bm[rr >> 5], 1u << (rr & 31));
          ++n_match;
        }
        const bool lit = valid && leader && !match;
        const unsigned litm = __ballot_sync(0xffffffffu, lit);
        if (lit) lits[nlw + __popc(litm & below)] = (uint16_t)rr;
        nlw += __popc(litm);
      }
    };
    uint4 rv0[kGV][kUPL], rv1[kGV][kUPL];
    load_refs(0, rv0);
#pragma unroll 1
    for (int g0 = 0; g0 < kStepsV; g0 += 2 * kGV) {
      if (g0 + kGV < kStepsV) load_refs(g0 + kGV, rv1);
      test(g0, rv0);
      if (g0 + kGV < kStepsV) {
        if (g0 + 2 * kGV < kStepsV) load_refs(g0 + 2 * kGV, rv0);
        test(g0 + kGV, rv1);
      }
    }
    __syncwarp();
    // ---- then the literal rows' codes into the warp's histogram, kLPR lanes per row, 4 codes each ----
    for (int i0 = 0; i0 < nlw; i0 += G::kRPS) {
      const int li = i0 + lane / G::kLPR;
      if (li < nlw) {
        const int rr = lits[li];
#pragma unroll
        for (int j = 0; j < G::kSPR; ++j) {
          const Quad wb = sm_quad(s_sym, (rr * (D / 4) + (lane % G::kLPR) + j * 32) * W, (Quad*)nullptr);
#pragma unroll
          for (int q = 0; q < 4; ++q) atomicAdd(&hist[quad_code(wb, q)], 1u);
        }
      }
    }
    n_lit = lane == 0 ? (uint32_t)nlw : 0u;
  } else {
    const unsigned gshift = lane & ~(G::kLPR - 1);
    const unsigned gmask = (G::kLPR == 32 ? 0xffffffffu : ((1u << G::kLPR) - 1u)) << gshift;
    const bool leader = (lane % G::kLPR) == 0;
      // the reference rows' codes of a group of steps (the next group's loads are in flight while
    // this one is compared)
    auto load_refs = [&](int g0, Quad (&wr)[kGroup][G::kSPR]) {
#pragma unroll
      for (int it = 0; it < kGroup; ++it) {
        const int rr = (warp * kSteps + g0 + it) * G::kRPS + lane / G::kLPR;
        const int64_t b = row0 + rr;
        const uint32_t ref = b < bend ? s_ref[rr] : (uint32_t)b;
#pragma unroll
        for (int j = 0; j < G::kSPR; ++j) {
          const int d = (lane % G::kLPR) * 4 + j * 128;
          wr[it][j] = ref != (uint32_t)b ? ld_quad(symt, (size_t)ref * D + d, (Quad*)nullptr) : Quad{};
        }
      }
    };
    auto process = [&](int g0, const Quad (&wr)[kGroup][G::kSPR]) {
#pragma unroll
      for (int it = 0; it < kGroup; ++it) {
        const int rr = (warp * kSteps + g0 + it) * G::kRPS + lane / G::kLPR;
        const int64_t b = row0 + rr;
        const bool valid = b < bend;
        const uint32_t ref = valid ? s_ref[rr] : 0u;
        const bool cand = valid && ref != (uint32_t)b;
        Quad wb[G::kSPR];
        bool eq = true;
#pragma unroll
        for (int j = 0; j < G::kSPR; ++j) {
          wb[j] = sm_quad(s_sym, so + (rr * (D / 4) + (lane % G::kLPR) + j * 32) * W, (Quad*)nullptr);
          bool e = quad_eq(wr[it][j], wb[j]);
          if (cand && e && quad_has_zero(wb[j])) {
            const int d = (lane % G::kLPR) * 4 + j * 128;
            const In* xb = x + ((size_t)b * T + t) * D + d;
            const In* xr = x + ((size_t)ref * T + t) * D + d;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (quad_code(wb[j], q) == 0u && raw32(xb[q]) != raw32(xr[q])) e = false;
          }
          eq = eq && e;
        }
        const unsigned bad = __ballot_sync(0xffffffffu, !eq);
        const bool match = cand && (bad & gmask) == 0u;
        if (valid && !match) {
#pragma unroll
          for (int j = 0; j < G::kSPR; ++j) {
#pragma unroll
            for (int q = 0; q < 4; ++q) atomicAdd(&hist[quad_code(wb[j], q)], 1u);
          }
        }
        if (valid && leader) {
          if (match) {
            w.ref[(size_t)t * B + b] = ref;
            atomicOr(&s_bm[rr >> 5], 1u << (rr & 31));
            ++n_match;
          } else {
            ++n_lit;
          }
        }
      }
    };
    Quad wr0[kGroup][G::kSPR], wr1[kGroup][G::kSPR];
    load_refs(0, wr0);
#pragma unroll 1
    for (int g0 = 0; g0 < kSteps; g0 += 2 * kGroup) {
      if (g0 + kGroup < kSteps) load_refs(g0 + kGroup, wr1);
      process(g0, wr0);
      if (g0 + kGroup < kSteps) {
        if (g0 + 2 * kGroup < kSteps) load_refs(g0 + 2 * kGroup, wr0);
        process(g0 + kGroup, wr1);
      }
    }
  }
  n_lit = __reduce_add_sync(0xffffffffu, n_lit);
  n_match = __reduce_add_sync(0xffffffffu, n_match);
  if (lane == 0) {
    atomicAdd(&s_cnt[0], n_lit);
    atomicAdd(&s_cnt[1], n_match);
  }
  __syncthreads();
#pragma unroll
  for (int i = tid; i < kA / 4; i += kNT) {   // four bins per thread and step
    uint4 f = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kNW; ++k) f = add4(f, reinterpret_cast<const uint4*>(s_histwin + k * kA)[i]);
    reinterpret_cast<uint4*>(w.seg_hist + (size_t)seg * kA)[i] = f;
    if (i == 0) s_cnt[2] = f.x;   // the literal rows' outliers: their codes of symbol 0
    uint32_t* th = w.tab_hist + (size_t)u * kA + 4 * i;
    if (f.x) atomicAdd(th + 0, f.x);
    if (f.y) atomicAdd(th + 1, f.y);
    if (f.z) atomicAdd(th + 2, f.z);
    if (f.w) atomicAdd(th + 3, f.w);
  }
  for (int i = tid; i < G::kBmWords; i += kNT) {   // bit i of word k: row b0 + 32 k + i of the slice
    const int64_t wi = (int64_t)s * G::kBmWords + i;
    if (wi < sh.nw) w.bitmap[(size_t)u * sh.nw + wi] = s_bm[i];
  }
  if (tid == 0) {
    const uint32_t chunks = (s_cnt[0] + G::kKC - 1) / G::kKC;
    w.seg_cnt[seg] = make_uint4(s_cnt[0], s_cnt[1], s_cnt[2], chunks);
    atomicAdd(&w.tab_cnt[u].x, s_cnt[0]);
    atomicAdd(&w.tab_cnt[u].y, s_cnt[1]);
    atomicAdd(&w.tab_cnt[u].z, s_cnt[2]);
    atomicAdd(&w.tab_cnt[u].w, chunks);
  }
}

// ---------------------------------------------------------------------------
// Block-wide helpers over 256 threads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  uint32_t tot = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += s_red[i];
  __syncthreads();
  return tot;
}

__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ void st_u64(uint8_t* p, unsigned long long v) {
  *reinterpret_cast<unsigned long long*>(p) = v;
}
__device__ __forceinline__ unsigned long long pad16(unsigned long long n) { return (n + 15ull) & ~15ull; }

// Completes the containers, run by the whole CTA (the last one of k_codebook,
// or of k_layout when the bitstream sizes come from there).  Thread r < R
// brings container r's counts, bitstream words and first-unit bases in c; this
// lays out its sections (a container is the single-call format for the rows
// of its slice), places the containers back to back (a scan of their sizes),
// writes the headers, zeroes the section padding and, for an empty batch, the
// table records (k_emit writes them otherwise), and sets the status.
__device__ void finish_containers(const Shape& sh, const EbParams& ep, const Work& w, ContLay c, uint8_t* out,
                                  unsigned long long cap, unsigned long long* out_bytes,
                                  unsigned long long* chunk_off, uint32_t epoch, uint32_t cabort) {
  __shared__ unsigned long long s_size[kMaxSlices];
  __shared__ unsigned long long s_sum[5];   // literals, matches, outliers, chunks, words
  __shared__ unsigned long long s_total;
  const int tid = threadIdx.x;
  const int T = sh.T;
  Glob* g = w.glob;
  if (tid < 5) s_sum[tid] = 0ull;
  __syncthreads();
  if (tid < sh.R) {
    const int64_t n = slice_rows(sh, tid);
    const unsigned long long nseg_r = (unsigned long long)div_up(n, sh.SB);
    const unsigned long long nw_r = (unsigned long long)div_up(n, 32);
    c.ref_bytes = (uint32_t)ref_bytes_of(n, sh.window);
    c.off_seg = kHeaderBytes + (unsigned long long)T * table_rec_bytes(sh.A);
    c.off_bitmap = c.off_seg + (unsigned long long)T * nseg_r * kSegRecBytes;
    c.off_chunks = c.off_bitmap + pad16((unsigned long long)T * nw_r * 4ull);
    c.off_refs = c.off_chunks + pad16(c.n_chunks * 2ull);
    c.off_bits = c.off_refs + pad16(c.n_match * c.ref_bytes);
    c.total = c.off_bits + 4ull * c.words;
    s_size[tid] = c.total;
    atomicAdd(&s_sum[0], c.n_lit);
    atomicAdd(&s_sum[1], c.n_match);
    atomicAdd(&s_sum[2], c.n_out);
    atomicAdd(&s_sum[3], c.n_chunks);
    atomicAdd(&s_sum[4], c.words);
  }
  __syncthreads();
  if (tid == 0) {   // container bases (every size is a multiple of 16 bytes)
    unsigned long long acc = 0;
    for (int r = 0; r < sh.R; ++r) {
      const unsigned long long v = s_size[r];
      s_size[r] = acc;
      acc += v;
    }
    s_total = acc;
  }
  __syncthreads();
  const unsigned long long total = s_total;
  int status = total > cap ? EBC_ERR_CAPACITY : EBC_OK;
  if (cabort == status_word(epoch, EBC_ERR_DEVICE_TIMEOUT)) status = EBC_ERR_DEVICE_TIMEOUT;
  if (tid < sh.R) {
    c.base = s_size[tid];
    w.cont[tid] = c;
    if (chunk_off) chunk_off[tid] = c.base;
    uint8_t* o = out + c.base;
    const int64_t n = slice_rows(sh, tid);
    if (c.base + kHeaderBytes <= cap) {
      st_u32(o + 0, kMagic); st_u32(o + 4, kFormatVersion); st_u64(o + 8, (unsigned long long)n);
      st_u32(o + 16, (uint32_t)T); st_u32(o + 20, (uint32_t)sh.D); st_u32(o + 24, (uint32_t)(sh.A / 2));
      st_u32(o + 28, kLmax); st_u32(o + 32, (uint32_t)sh.SB); st_u32(o + 36, (uint32_t)sh.KC);
      st_u32(o + 40, c.ref_bytes); st_u32(o + 44, (uint32_t)sh.window);
      st_u64(o + 48, c.n_lit); st_u64(o + 56, c.n_match); st_u64(o + 64, c.n_out); st_u64(o + 72, c.n_chunks);
      st_u64(o + 88, c.off_seg); st_u64(o + 96, c.off_bitmap); st_u64(o + 104, c.off_chunks);
      st_u64(o + 112, c.off_refs); st_u64(o + 120, c.off_bits); st_u64(o + 136, 0ull);
      if (status == EBC_OK) {
        st_u64(o + 80, c.words);
        st_u64(o + 128, c.total);
      }
    }
    if (status == EBC_OK) {   // the alignment padding after each variable-length section
      const unsigned long long bm_end = c.off_bitmap + (unsigned long long)T * (unsigned long long)div_up(n, 32) * 4ull;
      for (unsigned long long i = bm_end; i < c.off_chunks; ++i) o[i] = 0;
      for (unsigned long long i = c.off_chunks + c.n_chunks * 2ull; i < c.off_refs; ++i) o[i] = 0;
      for (unsigned long long i = c.off_refs + c.n_match * c.ref_bytes; i < c.off_bits; ++i) o[i] = 0;
    }
  }
  if (sh.nseg == 0 && status == EBC_OK) {   // an empty batch: every table record is eb and zeros
    const int per = (int)(table_rec_bytes(sh.A) / 4);
    const long long nrec = (long long)sh.R * T * per;
    for (long long i = tid; i < nrec; i += blockDim.x) {
      const int r = (int)(i / ((long long)T * per));
      const int t = (int)((i / per) % T);
      const int k = (int)(i % per);
      uint32_t* rec = reinterpret_cast<uint32_t*>(out + s_size[r] + kHeaderBytes + (size_t)t * (per * 4));
      rec[k] = k == 0 ? __float_as_uint(ep.eb[t]) : 0u;
    }
  }
  if (tid == 0) {
    g->n_lit = s_sum[0]; g->n_match = s_sum[1]; g->n_out = s_sum[2]; g->n_chunks = s_sum[3];
    g->words = s_sum[4];
    g->total = total;
    *out_bytes = total;
    if (status != EBC_OK) record_error(g, status);
    g->cstat = status_word(epoch, status);
    g->done = 0u;
  }
}

// The code of one unit over the wide alphabet (1024 symbols, 4 per thread):
// the same construction as for 256 symbols (two-queue Huffman over the leaves
// sorted by (count, symbol), ties to the leaf, halving above 24 bits;
// canonical values by the DEFLATE rule), with the leaf order and the canonical
// ranks counted per length (canonical_ranks).  Writes tabcode, tab_bits, tab_rec.
__device__ void huffman_wide(const Shape& sh, const EbParams& ep, const Work& w, int u, int t, bool raw,
                             uint32_t* s_f, uint32_t* s_lw, uint32_t* s_nodew, unsigned long long* s_key,
                             uint16_t* s_order, uint16_t* s_leafpar, uint16_t* s_nodepar, uint16_t* s_depth,
                             uint8_t* s_len, uint32_t* s_count, uint32_t* s_next, uint32_t* s_wcnt,
                             uint32_t* s_run, unsigned long long* s_bits64, int* s_maxlen, uint4* s_warp) {
  constexpr int kA = Alph<2>::kA, kPer = kA / 256;
  const int tid = threadIdx.x;
  uint32_t f0[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int sy = k * 256 + tid;
    // (with no segments, k_quantize did not run and the accumulators are stale)
    f0[k] = sh.nseg > 0 ? __ldcg(&w.tab_hist[(size_t)u * kA + sy]) : 0u;
    s_f[sy] = f0[k];
    s_len[sy] = raw ? (uint8_t)Alph<2>::kRawLen : 0;
  }
  __syncthreads();
  for (int round = 0; round < 40 && !raw; ++round) {
    if (tid == 0) *s_maxlen = 0;
    unsigned long long key[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int sy = k * 256 + tid;
      const uint32_t fi = s_f[sy];
      key[k] = fi > 0u ? ((unsigned long long)fi << 10) | (unsigned)sy : ~0ull;
      s_len[sy] = 0;
    }
    const int n = sort_used_keys<kPer>(key, s_key, s_warp);   // leaves in (count, symbol) order
    for (int i = tid; i < n; i += 256) {
      s_order[i] = (uint16_t)(s_key[i] & 1023u);
      s_lw[i] = (uint32_t)(s_key[i] >> 10);
    }
    __syncthreads();
    if (tid == 0 && n >= 2) {   // the two queues: leaves in order, merged nodes first in first out
      constexpr uint32_t kNone = 0xFFFFFFFFu;
      int li = 0, qi = 0, qn = 0;
      uint32_t a0 = s_lw[0], a1 = s_lw[1], q0 = kNone, q1 = kNone;
      for (int m = 0; m < n - 1; ++m) {
        uint32_t wsum = 0;
#pragma unroll
        for (int pick = 0; pick < 2; ++pick) {
          if (a0 <= q0) {   // a leaf (ties go to the leaf)
            s_leafpar[li] = (uint16_t)m;
            wsum += a0;
            ++li;
            a0 = a1;
            a1 = li + 1 < n ? s_lw[li + 1] : kNone;
          } else {
            s_nodepar[qi] = (uint16_t)m;
            wsum += q0;
            ++qi;
            q0 = q1;
            q1 = qi + 1 < qn ? s_nodew[qi + 1] : kNone;
          }
        }
        s_nodew[qn] = wsum;
        if (qn == qi) q0 = wsum;
        else if (qn == qi + 1) q1 = wsum;
        ++qn;
      }
    }
    __syncthreads();
    for (int m = tid; m < n - 1; m += 256) {   // depth of each merged node: walk up to the root (node n-2)
      int a = m, d = 0;
      while (a != n - 2) {
        a = s_nodepar[a];
        ++d;
      }
      s_depth[m] = (uint16_t)d;
    }
    __syncthreads();
    if (n == 1 && tid == 0) {
      s_len[s_order[0]] = 1;
      *s_maxlen = 1;
    }
    if (n >= 2)
      for (int i = tid; i < n; i += 256) {
        const int l = s_depth[s_leafpar[i]] + 1;
        s_len[s_order[i]] = (uint8_t)(l < 255 ? l : 255);
        atomicMax(s_maxlen, l);
      }
    __syncthreads();
    if (*s_maxlen <= kLmax) break;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int sy = k * 256 + tid;
      const uint32_t fi = s_f[sy];
      if (fi > 0u) s_f[sy] = (fi >> 1) > 0u ? (fi >> 1) : 1u;
    }
    __syncthreads();
  }
  // canonical codes: counts per length, first code and first rank of each length, then each
  // symbol's rank among its length from a sort by (length, symbol)
  if (tid < kLmax + 2) s_count[tid] = 0;
  __syncthreads();
  uint32_t lens[kPer], rk[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    lens[k] = s_len[k * 256 + tid];
    if (lens[k]) atomicAdd(&s_count[lens[k]], 1u);
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t c = 0;
    s_count[0] = 0;
    for (int l = 1; l <= kLmax; ++l) {
      c = (c + s_count[l - 1]) << 1;
      s_next[l] = c;
    }
  }
  canonical_ranks<kPer>(lens, rk, s_wcnt, s_run);
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    s_lw[k * 256 + tid] = lens[k] ? ((s_next[lens[k]] + rk[k]) << 8) | lens[k] : 0u;
  __syncthreads();
  unsigned long long sum = 0;   // bits of the unit's literal codes, plus the raw bits of its outliers
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int sy = k * 256 + tid;
    const uint32_t e = s_lw[sy];
    w.tabcode[(size_t)u * kA + sy] = e;
    sum += (unsigned long long)f0[k] * (e & 0xffu) + (sy == 0 ? 32ull * f0[k] : 0ull);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if ((tid & 31) == 0) s_bits64[tid >> 5] = sum;
  __syncthreads();
  if (tid == 0) {
    unsigned long long tot = 0;
    for (int k = 0; k < 8; ++k) tot += s_bits64[k];
    w.tab_bits[u] = tot;
    const uint4 tc = sh.nseg > 0 ? __ldcg(&w.tab_cnt[u]) : make_uint4(0, 0, 0, 0);
    w.tab_rec[u] = make_uint4(__float_as_uint(ep.eb[t]), tc.x, tc.y, tc.z);   // head of the table record
  }
}

// ---------------------------------------------------------------------------
// k_codebook: one CTA per unit.  Huffman code lengths (§III-D "Optimized
// Entropy Encoding") by the two-queue construction over leaves sorted by
// (count, symbol), merged nodes in FIFO order, ties to the leaf; if the longest
// code exceeds 24 bits every nonzero count becomes max(1, count >> 1) and the
// code is rebuilt.  Canonical code values follow the DEFLATE rule.  The last
// CTA to finish lays out the containers and writes their headers.
// ---------------------------------------------------------------------------
template <int W>
__global__ void __launch_bounds__(256) k_codebook(Shape sh, EbParams ep, Work w, uint8_t* __restrict__ out,
                                                   unsigned long long cap, unsigned long long* out_bytes,
                                                   unsigned long long* chunk_off, uint32_t epoch) {
  pdl_enter();
  constexpr int kA = Alph<W>::kA;
  using Par = typename std::conditional<W == 1, uint8_t, uint16_t>::type;   // node indices and depths
  __shared__ uint32_t s_f[kA], s_lw[kA], s_nodew[kA];
  __shared__ unsigned long long s_key[kA];
  __shared__ uint4 s_seg[kFoldMaxSeg];
  __shared__ unsigned long long s_bits64[8];
  __shared__ uint16_t s_order[kA];
  __shared__ Par s_leafpar[kA], s_nodepar[kA], s_depth[kA];
  __shared__ __align__(16) uint8_t s_len[kA];
  __shared__ uint32_t s_count[kLmax + 2], s_next[kLmax + 2], s_run[kLmax + 2];
  __shared__ int s_maxlen, s_last;
  __shared__ uint32_t s_wn[8];                // used symbols per warp
  __shared__ uint32_t s_wcnt[8][kLmax + 1];   // symbols of each length per warp
  __shared__ uint4 s_warp[8];
  __shared__ uint4 s_cpre[kMaxSlices + 1], s_wpre[kMaxSlices + 1];   // unit prefixes at container starts
  const int tid = threadIdx.x;
  const int u = blockIdx.x;   // unit: slice u / T, table u % T
  const int T = sh.T;
  const int U = sh.U;
  Glob* g = w.glob;

  if (u < U && sh.fold && sh.nseg > 0) {
    // the segments' chunk and match counts (nseg <= 256), requested before the code is built
    if (tid < sh.nseg) {
      const uint4 cnt = __ldcg(&w.seg_cnt[u * sh.nseg + tid]);
      s_seg[tid] = make_uint4(0u, cnt.w, cnt.y, 0u);
    }
  }
  if (u < U) {
    const int t = u % T;
    const bool raw = (table_mode(w, t) & kModeRawCodes) != 0;   // every code log2(A) bits: no Huffman
    if constexpr (W == 2) {
      huffman_wide(sh, ep, w, u, t, raw, s_f, s_lw, s_nodew, s_key, s_order, s_leafpar, s_nodepar, s_depth, s_len,
                   s_count, s_next, &s_wcnt[0][0], s_run, s_bits64, &s_maxlen, s_warp);
    } else {
    // (with no segments, k_quantize did not run and the accumulators are stale)
    const uint32_t f0 = sh.nseg > 0 ? __ldcg(&w.tab_hist[(size_t)u * 256 + tid]) : 0u;
    const uint4 tc = tid == 0 && sh.nseg > 0 ? __ldcg(&w.tab_cnt[u]) : make_uint4(0, 0, 0, 0);
    s_f[tid] = f0;
    if (raw) s_len[tid] = 8;
    __syncthreads();
    for (int round = 0; round < 40 && !raw; ++round) {
      const uint32_t fi = s_f[tid];
      // leaves in (count, symbol) order: the keys count << 8 | symbol of the used symbols are
      // compacted, and each is placed at its rank among them (the keys are distinct)
      const int lane = tid & 31, wp = tid >> 5;
      const unsigned used = __ballot_sync(0xffffffffu, fi > 0u);
      if (lane == 0) s_wn[wp] = __popc(used);
      __syncthreads();
      int n = 0, pos = __popc(used & ((1u << lane) - 1u));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pos += k < wp ? (int)s_wn[k] : 0;
        n += (int)s_wn[k];
      }
      if (fi > 0u) s_key[pos] = ((unsigned long long)fi << 8) | (unsigned)tid;
      __syncthreads();
      if (tid < n) {
        const unsigned long long mk = s_key[tid];
        int rank = 0;
#pragma unroll 4
        for (int j = 0; j < n; ++j) rank += s_key[j] < mk ? 1 : 0;
        s_order[rank] = (uint16_t)(mk & 0xffu);
        s_lw[rank] = (uint32_t)(mk >> 8);
      }
      s_len[tid] = 0;
      if (tid == 0) s_maxlen = 0;
      __syncthreads();
      if (tid == 0 && n >= 2) {
        // the heads of both queues and the entries after them live in
        // registers (kNone = exhausted), so a pick is a compare and a few moves
        constexpr uint32_t kNone = 0xFFFFFFFFu;   // above any weight (the sum of all counts is < 2^32)
        int li = 0, qi = 0, qn = 0;
        uint32_t a0 = s_lw[0], a1 = s_lw[1], q0 = kNone, q1 = kNone;
        for (int m = 0; m < n - 1; ++m) {
          uint32_t wsum = 0;
#pragma unroll
          for (int pick = 0; pick < 2; ++pick) {
            if (a0 <= q0) {   // a leaf (ties go to the leaf)
              s_leafpar[li] = (uint8_t)m;
              wsum += a0;
              ++li;
              a0 = a1;
              a1 = li + 1 < n ? s_lw[li + 1] : kNone;
            } else {
              s_nodepar[qi] = (uint8_t)m;
              wsum += q0;
              ++qi;
              q0 = q1;
              q1 = qi + 1 < qn ? s_nodew[qi + 1] : kNone;
            }
          }
          s_nodew[qn] = wsum;
          if (qn == qi) q0 = wsum;
          else if (qn == qi + 1) q1 = wsum;
          ++qn;
        }
      }
      __syncthreads();
      if (n >= 2 && tid < n - 1) {   // depth of each merged node: walk up to the root (node n-2)
        int m = tid, d = 0;
        while (m != n - 2) {
          m = s_nodepar[m];
          ++d;
        }
        s_depth[tid] = (uint8_t)d;
      }
      __syncthreads();
      if (n == 1 && tid == 0) {
        s_len[s_order[0]] = 1;
        s_maxlen = 1;
      }
      if (n >= 2 && tid < n) {
        const int l = s_depth[s_leafpar[tid]] + 1;
        s_len[s_order[tid]] = (uint8_t)l;
        atomicMax(&s_maxlen, l);
      }
      __syncthreads();
      if (s_maxlen <= kLmax) break;
      if (fi > 0u) s_f[tid] = (fi >> 1) > 0u ? (fi >> 1) : 1u;
      __syncthreads();
    }
    // canonical codes: counts per length, and each symbol's rank among the symbols of its length
    // below it (in its warp by a match mask, in the warps before by their counts)
    const int lane = tid & 31, wp = tid >> 5;
    if (tid < kLmax + 2) s_count[tid] = 0;
    for (int i = tid; i < 8 * (kLmax + 1); i += 256) (&s_wcnt[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t L = s_len[tid];
    if (L) atomicAdd(&s_count[L], 1u);
    const unsigned same = __match_any_sync(0xffffffffu, L);
    if (lane == __ffs(same) - 1) s_wcnt[wp][L] = (uint32_t)__popc(same);
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
      code = s_next[L] + (uint32_t)__popc(same & ((1u << lane) - 1u));
      for (int k = 0; k < wp; ++k) code += s_wcnt[k][L];
    }
    w.tabcode[(size_t)u * 256 + tid] = (code << 8) | L;
    {   // bits of the table's literal codes, plus the raw bits of its outliers (symbol 0)
      unsigned long long sum = (unsigned long long)f0 * L + (tid == 0 ? 32ull * f0 : 0ull);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if ((tid & 31) == 0) s_bits64[tid >> 5] = sum;
      __syncthreads();
      if (tid == 0) {
        unsigned long long tot = 0;
        for (int k = 0; k < 8; ++k) tot += s_bits64[k];
        w.tab_bits[u] = tot;
        w.tab_rec[u] = make_uint4(__float_as_uint(ep.eb[t]), tc.x, tc.y, tc.z);   // head of the table record
      }
    }
    }   // W == 1
    if (sh.fold && sh.nseg > 0) {
      // this unit's segments: bits = sum over codes of count * length (+32 raw bits per outlier),
      // one warp per segment, eight histograms in flight per warp (lengths from shared memory);
      // then offsets relative to the unit (a scan) and the unit's totals
      const int warp = tid >> 5, lane = tid & 31;
      constexpr int kV = kA / 128;                  // uint4 of histogram (and words of 4 lengths) per lane
      constexpr int kBatch = W == 1 ? 8 : 2;        // segments per warp whose histograms are loaded together
                                                    // (more would keep two CTAs of 256 threads off an SM)
      __syncthreads();   // the unit's code lengths are final
      uint32_t c[kV];
#pragma unroll
      for (int v = 0; v < kV; ++v) c[v] = reinterpret_cast<const uint32_t*>(s_len)[lane * kV + v];
      for (int i0 = warp; i0 < sh.nseg; i0 += 8 * kBatch) {
        uint4 h[kBatch][kV];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = i0 + 8 * q;
          if (i < sh.nseg) {
            const uint4* hp = reinterpret_cast<const uint4*>(w.seg_hist + (size_t)(u * sh.nseg + i) * kA) + lane * kV;
#pragma unroll
            for (int v = 0; v < kV; ++v) h[q][v] = __ldcg(hp + v);
          }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = i0 + 8 * q;
          if (i < sh.nseg) {
            uint32_t bits = 0;
#pragma unroll
            for (int v = 0; v < kV; ++v)
              bits += h[q][v].x * (c[v] & 0xffu) + h[q][v].y * ((c[v] >> 8) & 0xffu) +
                      h[q][v].z * ((c[v] >> 16) & 0xffu) + h[q][v].w * (c[v] >> 24);
            if (lane == 0) bits += 32u * h[q][0].x;   // symbol 0: the outliers' raw bits
            bits = __reduce_add_sync(0xffffffffu, bits);
            if (lane == 0) {
              s_seg[i].x = ((bits + 127u) >> 7) * 4u;
              s_seg[i].w = bits;
            }
          }
        }
      }
      __syncthreads();
      uint4 v = tid < sh.nseg ? s_seg[tid] : make_uint4(0, 0, 0, 0);
      const uint32_t segbits = v.w;
      v.w = 0;
      uint4 tot;
      const uint4 ex = block_excl_scan4(v, &tot, s_warp);
      if (tid < sh.nseg) w.seg_base[u * sh.nseg + tid] = make_uint4(ex.x, ex.y, ex.z, segbits);
      if (tid == 0) w.seg_desc[u] = tot;
    }
  }

  // ---- the last CTA: container layouts and headers ----
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&g->done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const uint32_t cab = __ldcg(&g->cabort);   // (read now: the status needs it at the end)
  // exclusive scans over the units of their counts (and, folded, of their bitstream sizes); the
  // values at each container's first unit, and the totals, are kept
  const bool have = sh.nseg > 0;
  for (int i = tid; i <= sh.R; i += 256) s_cpre[i] = s_wpre[i] = make_uint4(0, 0, 0, 0);   // (T = 0: no units)
  __syncthreads();
  uint4 carry = make_uint4(0, 0, 0, 0), wcarry = make_uint4(0, 0, 0, 0);
  for (int base = 0; base < U; base += 256) {
    const int i = base + tid;
    const uint4 v = i < U && have ? __ldcg(&w.tab_cnt[i]) : make_uint4(0, 0, 0, 0);
    const uint4 d = i < U && have && sh.fold ? __ldcg(&w.seg_desc[i]) : make_uint4(0, 0, 0, 0);
    uint4 tot;
    const uint4 ex = add4(carry, block_excl_scan4(v, &tot, s_warp));
    if (i < U && i % T == 0) s_cpre[i / T] = ex;
    carry = add4(carry, tot);
    if (sh.fold && have) {
      const uint4 wex = add4(wcarry, block_excl_scan4(d, &tot, s_warp));
      if (i < U) w.tile_base[i] = wex;
      if (i < U && i % T == 0) s_wpre[i / T] = wex;
      wcarry = add4(wcarry, tot);
    }
  }
  if (tid == 0) {
    s_cpre[sh.R] = carry;
    s_wpre[sh.R] = wcarry;
  }
  __syncthreads();
  ContLay c{};
  if (tid < sh.R) {
    const uint4 a = s_cpre[tid], b = s_cpre[tid + 1];
    c.n_lit = b.x - a.x;
    c.n_match = b.y - a.y;
    c.n_out = b.z - a.z;
    c.n_chunks = b.w - a.w;
    const uint4 wa = s_wpre[tid], wb = s_wpre[tid + 1];
    c.words = wb.x - wa.x;   // folded (else completed by k_layout)
    c.word0 = wa.x;
    c.chunk0 = wa.y;
    c.match0 = wa.z;
  }
  if (sh.fold || !have) {
    finish_containers(sh, ep, w, c, out, cap, out_bytes, chunk_off, epoch, cab);
  } else {
    if (tid < sh.R) w.cont[tid] = c;   // the counts; k_layout adds the bitstream sizes
    if (tid == 0) {
      g->cstat = status_word(epoch, EBC_OK);
      g->done = 0u;
    }
  }
}

// ORs the n (1..64) right-aligned bits of str MSB-first into a word array at bit
// position p (up to three words).
__device__ __forceinline__ void put_string(uint32_t* s, uint32_t p, unsigned long long str, uint32_t n) {
  const unsigned long long v = str << (64u - n);   // left-aligned
  const uint32_t sh = p & 31u;
  uint32_t* w = s + (p >> 5);
  const unsigned long long hi = v >> sh;
  atomicOr(w, (uint32_t)(hi >> 32));
  if (sh + n > 32u) atomicOr(w + 1, (uint32_t)hi);
  if (sh + n > 64u) atomicOr(w + 2, (uint32_t)((v << (64u - sh)) >> 32));
}

// Writes `len` (1..32) bits of `code` MSB-first at bit position p of a word array.
__device__ __forceinline__ void put_bits(uint32_t* s, uint32_t p, uint32_t code, uint32_t len) {
  const uint32_t sh = p & 31u;
  const unsigned long long v = ((unsigned long long)code << (64u - len)) >> sh;
  atomicOr(&s[p >> 5], (uint32_t)(v >> 32));
  const uint32_t lo = (uint32_t)v;
  if (lo) atomicOr(&s[(p >> 5) + 1], lo);
}

// Rows of bitmap word wi of a segment that exist in the batch.
__device__ __forceinline__ uint32_t valid_mask(int64_t B, int64_t row0, int wi) {
  const int64_t nv = B - (row0 + (int64_t)wi * 32);
  return nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
}

// ---------------------------------------------------------------------------
// k_layout: per-segment aggregates.  One warp per segment computes its bit
// count (sum over codes of count * length, plus 32 raw bits per outlier) from
// its histogram; a CTA covers 8 consecutive segments and stores, per segment,
// {words, chunks, matches, bits} relative to the CTA's first segment and, per
// CTA, the totals.  The last CTA to finish turns the CTA totals into absolute
// bases (an exclusive scan) and completes the header (bitstream words, total
// size) and the capacity check.  No CTA waits on another.
// ---------------------------------------------------------------------------
template <int W>
__global__ void __launch_bounds__(256) k_layout(Shape sh, EbParams ep, Work w, uint8_t* __restrict__ out,
                                                 unsigned long long cap, unsigned long long* out_bytes,
                                                 unsigned long long* chunk_off, uint32_t epoch) {
  pdl_enter();
  __shared__ uint4 s_agg[8];
  __shared__ uint4 s_warp[8];
  __shared__ int s_last;
  Glob* g = w.glob;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const int ntiles = gridDim.x;
  const int nsegT = sh.U * sh.nseg;
  const int seg = tile * 8 + warp;
  uint4 a = make_uint4(0, 0, 0, 0);   // {words, chunks, matches, -}
  uint32_t bits = 0;
  if (seg < nsegT) {
    constexpr int kA = Alph<W>::kA, kV = kA / 128;   // uint4 of histogram and codes per lane
    const int u = seg / sh.nseg;
    const uint4* hp = reinterpret_cast<const uint4*>(w.seg_hist + (size_t)seg * kA) + lane * kV;
    const uint4* cp = reinterpret_cast<const uint4*>(w.tabcode + (size_t)u * kA) + lane * kV;
    const uint4 cnt = __ldcg(&w.seg_cnt[seg]);
    uint32_t h0x = 0;
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      const uint4 h = __ldcg(hp + v), c = __ldcg(cp + v);
      bits += h.x * (c.x & 0xffu) + h.y * (c.y & 0xffu) + h.z * (c.z & 0xffu) + h.w * (c.w & 0xffu);
      if (v == 0) h0x = h.x;
    }
    if (lane == 0) bits += 32u * h0x;   // symbol 0: the outliers' raw bits
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) bits += __shfl_xor_sync(0xffffffffu, bits, off);
    a = make_uint4(((bits + 127u) >> 7) * 4u, cnt.w, cnt.y, 0u);
  }
  if (lane == 0) s_agg[warp] = a;
  __syncthreads();
  if (seg < nsegT && lane == 0) {
    uint4 pre = make_uint4(0, 0, 0, 0);
    for (int i = 0; i < warp; ++i) pre = add4(pre, s_agg[i]);
    w.seg_base[seg] = make_uint4(pre.x, pre.y, pre.z, bits);   // relative to the tile; made absolute by k_emit
  }
  if (tid == 0) {
    uint4 tot = make_uint4(0, 0, 0, 0);
    for (int i = 0; i < 8; ++i) tot = add4(tot, s_agg[i]);
    w.seg_desc[tile] = tot;
  }
  // ---- the last CTA: exclusive scan of the CTA totals, header completion ----
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&g->done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint4 carry = make_uint4(0, 0, 0, 0);
  for (int base = 0; base < ntiles; base += 256) {
    const int i = base + tid;
    const uint4 v = i < ntiles ? __ldcg(&w.seg_desc[i]) : make_uint4(0, 0, 0, 0);
    uint4 tot;
    const uint4 ex = block_excl_scan4(v, &tot, s_warp);
    if (i < ntiles) w.tile_base[i] = add4(carry, ex);
    carry = add4(carry, tot);
  }
  __syncthreads();
  // each container's bitstream: the absolute bases at its first segment and after its last
  ContLay c{};
  if (tid < sh.R) {
    c = w.cont[tid];   // counts, from k_codebook
    uint4 at[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = (tid + e) * sh.T * sh.nseg;   // first segment of container tid + e
      if (i >= nsegT) {
        at[e] = carry;
      } else {
        const uint4 tb = __ldcg(&w.tile_base[i >> 3]), rel = __ldcg(&w.seg_base[i]);
        at[e] = make_uint4(tb.x + rel.x, tb.y + rel.y, tb.z + rel.z, 0u);
      }
    }
    c.words = at[1].x - at[0].x;
    c.word0 = at[0].x;
    c.chunk0 = at[0].y;
    c.match0 = at[0].z;
  }
  finish_containers(sh, ep, w, c, out, cap, out_bytes, chunk_off, epoch, __ldcg(&w.glob->cabort));
}

// ---------------------------------------------------------------------------
// k_emit: one CTA per (unit, segment), offsets from k_codebook or k_layout.  Every global
// read the CTA needs (the segment's codes, into shared memory; bitmap,
// references, code table) is issued first.  The literal rows are ranked from
// the match bitmap and dealt to the warps in turn (kRPS rows per warp step,
// kLPR lanes per row, 4 codes per lane), so matched rows cost nothing and the
// warps get even shares.  Pass 1 adds up each literal row's code lengths; a
// scan over the ranks gives each row's bit offset; in pass 2 each lane joins
// its codes into one bit string that is ORed into a shared-memory copy of the
// segment's bitstream at the lane's offset (a prefix sum over the row).
// Outlier codes are followed by the 32 raw bits of the value.  The copy is
// stored with 16-byte writes; a segment larger than the copy (16 bits per
// code of the segment on average, reached only by outlier-heavy rows) is ORed
// straight into the zeroed output.  128 threads: a segment holds few literal
// rows (most rows are matches), so the per-segment work (code table, bitmap,
// ranks, scans) dominates and is cheaper on a smaller CTA.
// ---------------------------------------------------------------------------
constexpr int kET = 128, kEW = kET / 32;
template <int D>
constexpr int emit_stage_bytes() { return Geo<D>::kSegSyms * 2; }
template <int D, typename In, int W>
__global__ void __launch_bounds__(kET, 8) k_emit(const In* __restrict__ x, Shape sh, Work w,
                                               uint8_t* __restrict__ out, unsigned long long cap, uint32_t epoch) {
  pdl_enter();
  using G = Geo<D>;
  using Quad = typename QuadOf<W>::T;
  constexpr int kA = Alph<W>::kA;
  constexpr int kRPT = (G::kSB + kET - 1) / kET;   // rows (and ranks) per thread
  constexpr uint32_t kSmemWords = (uint32_t)emit_stage_bytes<D>() / 4u;
  extern __shared__ __align__(16) uint32_t s_bits[];
  __shared__ __align__(16) uint32_t s_sym[G::kSegSyms * W / 4 + 4];   // the segment's codes, row-major
  __shared__ uint32_t s_code[kA];
  __shared__ uint32_t s_bm[G::kBmWords];      // match bits
  __shared__ uint32_t s_lit[G::kBmWords];     // literal bits
  __shared__ uint32_t s_pre[G::kBmWords];     // literal (low 16) and match (high 16) rows before each word
  __shared__ uint32_t s_rowoff[G::kSB + 1];   // by literal rank: bits, then bit offset
  __shared__ uint16_t s_litrow[G::kSB];       // by literal rank: row
  __shared__ uint4 s_warp[8];
  Glob* g = w.glob;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // segment s of unit u = (slice r, table t): rows lrow0 .. of the slice, b0 + lrow0 .. of the batch
  const int seg = blockIdx.x;
  const int u = seg / sh.nseg;
  const int s = seg - u * sh.nseg;
  const int r = u / sh.T;
  const int t = u - r * sh.T;
  const int T = sh.T;
  const int64_t b0 = slice_row0(sh, r);
  const int64_t nr = slice_rows(sh, r);                     // rows of the slice
  const int64_t lrow0 = (int64_t)s * G::kSB;
  const int64_t row0 = b0 + lrow0;
  const int nseg_r = div_up(nr, G::kSB), nw_r = div_up(nr, 32);
  const uint8_t* symt = w.sym + (size_t)t * sh.symstride;
  // word offset of the codes in s_sym (even when W = 2)
  const int so = D * W >= 16 ? 0 : (int)(((size_t)row0 * D * W) & 15u) / 4;

  // ---- every global read, issued together ----
  {   // the dedup tables are not read again: empty them for the next call (a share per CTA)
    const unsigned long long n2 = (unsigned long long)sh.U * sh.S / 2;   // slot pairs (S is even)
    const unsigned long long per = (n2 + gridDim.x - 1) / gridDim.x;
    const unsigned long long lo = per * blockIdx.x, hi = lo + per < n2 ? lo + per : n2;
    uint4* sl = reinterpret_cast<uint4*>(w.slots);
    for (unsigned long long i = lo + tid; i < hi; i += kET) sl[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
  }
  const bool writable = __ldcg(&g->cstat) == status_word(epoch, EBC_OK);
  const ContLay cl = w.cont[r];
  uint32_t mycode[kA / kET];
#pragma unroll
  for (int k = 0; k < kA / kET; ++k) mycode[k] = __ldcg(&w.tabcode[(size_t)u * kA + k * kET + tid]);
  if (s == 0 && writable) {   // the unit's table record: eb, counts, code lengths
    uint8_t* rec = out + cl.base + kHeaderBytes + (size_t)t * Alph<W>::kRecBytes;
#pragma unroll
    for (int k = 0; k < kA / kET; ++k) rec[16 + k * kET + tid] = (uint8_t)(mycode[k] & 0xffu);
    if (tid == 0) *reinterpret_cast<uint4*>(rec) = __ldcg(&w.tab_rec[u]);
  }
  if (s >= nseg_r) return;   // past the end of a shorter slice: no rows
  const uint4 sbr = __ldcg(&w.seg_base[seg]);       // {words, chunks, matches} within its group, bits
  const uint4 tb = __ldcg(&w.tile_base[sh.fold ? u : seg >> 3]);   // absolute base of its group
  // the segment's bases within its container
  const uint4 sb = make_uint4(tb.x + sbr.x - cl.word0, tb.y + sbr.y - cl.chunk0, tb.z + sbr.z - cl.match0, sbr.w);
  uint32_t bmw = 0;
  if (tid < G::kBmWords) {
    const int64_t wi = (int64_t)s * G::kBmWords + tid;
    bmw = wi < sh.nw ? __ldcg(&w.bitmap[(size_t)u * sh.nw + wi]) : 0u;
  }
  {   // rows row0 .. row0 + SB are contiguous; the table stride is padded to 16 bytes
    const int64_t nrows = nr - lrow0 < G::kSB ? nr - lrow0 : G::kSB;
    const int nq = (int)((so * 4 + nrows * D * W + 15) / 16);
    const uint4* src = reinterpret_cast<const uint4*>(symt + (size_t)row0 * D * W - so * 4);
    uint4* dst = reinterpret_cast<uint4*>(s_sym);
    for (int i = tid; i < nq; i += kET) dst[i] = __ldcg(src + i);
  }
  uint32_t refw[kRPT];
#pragma unroll
  for (int k = 0; k < kRPT; ++k) {
    const int rr = k * kET + tid;
    refw[k] = (rr < G::kSB && lrow0 + rr < nr) ? __ldcg(&w.ref[(size_t)t * sh.B + row0 + rr]) : 0u;
  }
  const unsigned long long cbase = cl.base;
  const unsigned long long off_bits = cbase + cl.off_bits, off_chunks = cbase + cl.off_chunks;
  const unsigned long long off_refs = cbase + cl.off_refs;
  const unsigned long long off_seg = cbase + cl.off_seg, off_bitmap = cbase + cl.off_bitmap;
  const int ref_bytes = (int)cl.ref_bytes;

#pragma unroll
  for (int k = 0; k < kA / kET; ++k) s_code[k * kET + tid] = mycode[k];
  if (tid < G::kBmWords) {
    s_bm[tid] = bmw;
    s_lit[tid] = ~bmw & valid_mask(nr, lrow0, tid);
  }
  const uint32_t bits = sb.w;
  const uint32_t nwords = ((bits + 127u) >> 7) * 4u;
  const bool bits_fit = writable && off_bits + 4ull * ((unsigned long long)sb.x + nwords) <= cap;
  const bool in_smem = nwords <= kSmemWords;
  uint32_t* dstw = reinterpret_cast<uint32_t*>(out + off_bits) + sb.x;
  uint32_t* bitbuf = in_smem ? s_bits : dstw;
  if (bits_fit)
    for (uint32_t i = tid; i < nwords; i += kET) bitbuf[i] = 0u;
  __syncthreads();

  // ---- literal ranks: rows counted before each bitmap word, then each literal row's rank ----
  uint32_t nlit;
  {
    const uint32_t v = tid < G::kBmWords ? ((uint32_t)__popc(s_lit[tid]) | ((uint32_t)__popc(s_bm[tid]) << 16)) : 0u;
    uint4 tot;
    const uint4 ex = block_excl_scan4(make_uint4(v, 0, 0, 0), &tot, s_warp);
    if (tid < G::kBmWords) s_pre[tid] = ex.x;
    nlit = tot.x & 0xffffu;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kRPT; ++k) {
    const int rr = k * kET + tid;
    if (rr < G::kSB && ((s_lit[rr >> 5] >> (rr & 31)) & 1u))
      s_litrow[(s_pre[rr >> 5] & 0xffffu) + __popc(s_lit[rr >> 5] & ((1u << (rr & 31)) - 1u))] = (uint16_t)rr;
  }
  __syncthreads();
  const uint32_t nsteps = (nlit + G::kRPS - 1) / G::kRPS;

  // ---- pass 1: bits of each literal row ----
#pragma unroll 1
  for (uint32_t i = warp; i < nsteps; i += kEW) {
    const uint32_t k = i * G::kRPS + lane / G::kLPR;   // literal rank of this lane's row
    const bool act = k < nlit;
    const int rr = act ? s_litrow[k] : 0;
    uint32_t nb = 0;
#pragma unroll
    for (int j = 0; j < G::kSPR; ++j) {
      const Quad v = sm_quad(s_sym, so + (rr * (D / 4) + (lane % G::kLPR) + j * 32) * W, (Quad*)nullptr);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t c = quad_code(v, q);
        nb += act ? (s_code[c] & 0xffu) + (c == 0u ? 32u : 0u) : 0u;
      }
    }
    if constexpr (G::kLPR == 32) {
      nb = __reduce_add_sync(0xffffffffu, nb);
    } else {
#pragma unroll
      for (int off = G::kLPR / 2; off > 0; off >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, off);
    }
    if (act && (lane % G::kLPR) == 0) s_rowoff[k] = nb;
  }
  __syncthreads();

  // ---- bit offset of each literal row: scan over the ranks ----
  {
    uint4 loc[kRPT];
    uint4 sum = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const uint32_t kk = (uint32_t)(tid * kRPT + k);
      loc[k] = sum;
      if (kk < nlit) sum.x += s_rowoff[kk];
    }
    uint4 tot;
    const uint4 ex = block_excl_scan4(sum, &tot, s_warp);
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const uint32_t kk = (uint32_t)(tid * kRPT + k);
      if (kk < nlit) s_rowoff[kk] = ex.x + loc[k].x;
    }
    if (tid == 0) {
      s_rowoff[nlit] = tot.x;
      if (tot.x != bits) record_error(g, EBC_ERR_INTERNAL);
    }
  }
  __syncthreads();

  // ---- pass 2: codes (and raw outlier bits) into the bitstream ----
  if (bits_fit) {
#pragma unroll 1
    for (uint32_t i = warp; i < nsteps; i += kEW) {
      const uint32_t k = i * G::kRPS + lane / G::kLPR;
      const bool act = k < nlit;
      const int rr = act ? s_litrow[k] : 0;
      const int64_t b = row0 + rr;
      uint32_t p = act ? s_rowoff[k] : 0u;
#pragma unroll
      for (int j = 0; j < G::kSPR; ++j) {
        const Quad v = sm_quad(s_sym, so + (rr * (D / 4) + (lane % G::kLPR) + j * 32) * W, (Quad*)nullptr);
        // the lane's 4 codes joined into one string (right-aligned), if short and outlier-free
        uint32_t nb = 0;
        unsigned long long str = 0;
        bool plain = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t c = quad_code(v, q);
          const uint32_t e = s_code[c];
          const uint32_t len = e & 0xffu;
          str = (str << len) | (e >> 8);
          nb += len + (c == 0u ? 32u : 0u);
          plain = plain && c != 0u;
        }
        plain = plain && nb <= 64u;
        if (!act) nb = 0;
        uint32_t inc = nb;
#pragma unroll
        for (int off = 1; off < G::kLPR; off <<= 1) {
          const uint32_t n = __shfl_up_sync(0xffffffffu, inc, off);
          if ((lane % G::kLPR) >= off) inc += n;
        }
        const uint32_t slab_total = __shfl_sync(0xffffffffu, inc, (lane & ~(G::kLPR - 1)) + G::kLPR - 1);
        if (act && plain) {
          put_string(bitbuf, p + inc - nb, str, nb);
        } else if (act) {
          uint32_t qpos = p + inc - nb;
          const int d = (lane % G::kLPR) * 4 + j * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t c = quad_code(v, q);
            const uint32_t e = s_code[c];
            put_bits(bitbuf, qpos, e >> 8, e & 0xffu);
            qpos += e & 0xffu;
            if (c == 0u) {
              put_bits(bitbuf, qpos, raw32(x[((size_t)b * T + t) * D + d + q]), 32u);
              qpos += 32u;
            }
          }
        }
        p += slab_total;
      }
    }
  }
  __syncthreads();

  if (writable) {
    if (bits_fit && in_smem) {
      uint4* dst = reinterpret_cast<uint4*>(dstw);
      const uint4* src = reinterpret_cast<const uint4*>(s_bits);
      for (uint32_t i = tid; i < nwords / 4; i += kET) dst[i] = src[i];
    }
    for (uint32_t k = tid * G::kKC; k < nlit; k += kET * G::kKC) {
      const uint32_t end = k + G::kKC < nlit ? k + G::kKC : nlit;
      *reinterpret_cast<uint16_t*>(out + off_chunks + 2ull * (sb.y + k / G::kKC)) =
          (uint16_t)(s_rowoff[end] - s_rowoff[k]);
    }
#pragma unroll
    for (int k = 0; k < kRPT; ++k) {
      const int rr = k * kET + tid;
      if (rr < G::kSB && lrow0 + rr < nr && ((s_bm[rr >> 5] >> (rr & 31)) & 1u)) {
        const uint32_t mrank = (s_pre[rr >> 5] >> 16) + __popc(s_bm[rr >> 5] & ((1u << (rr & 31)) - 1u));
        const unsigned long long o = off_refs + (unsigned long long)ref_bytes * (sb.z + mrank);
        const uint32_t lref = refw[k] - (uint32_t)b0;   // the reference row within the slice
        if (sh.window) out[o] = (uint8_t)((uint32_t)(row0 + rr) - refw[k]);   // distance back, 1..window
        else if (ref_bytes == 2) *reinterpret_cast<uint16_t*>(out + o) = (uint16_t)lref;
        else *reinterpret_cast<uint32_t*>(out + o) = lref;
      }
    }
    if (tid == 0) {   // record t * nseg_r + s of the container
      uint32_t* rec = reinterpret_cast<uint32_t*>(out + off_seg + ((unsigned long long)t * nseg_r + s) * kSegRecBytes);
      rec[0] = sb.x; rec[1] = sb.y; rec[2] = sb.z; rec[3] = bits;
    }
    if (tid < G::kBmWords) {
      const int64_t wi = (int64_t)s * G::kBmWords + tid;
      if (wi < nw_r)
        *reinterpret_cast<uint32_t*>(out + off_bitmap + 4ull * ((size_t)t * nw_r + wi)) = s_bm[tid];
    }
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <int D, typename In, int W>
static void launch_compress_d(const In* x, const Shape& sh, const EbParams& ep, const Work& w, uint8_t* out,
                              unsigned long long cap, unsigned long long* out_bytes, unsigned long long* chunk_off,
                              uint32_t epoch, cudaStream_t st, Prof* prof, const CUtensorMap* xmap) {
  const unsigned grid = (unsigned)(sh.U * sh.nseg);          // (unit, segment) pairs
  const unsigned qsegs = (unsigned)(sh.T * sh.qseg);         // (table, segment) pairs of the whole batch
  if (grid) {
    // persistent quantize: as many CTAs as fit at once (two input stages each), at most one per segment
    static int per_sm = -1;
    const int smem = 2 * (int)QGeo<D, In>::kStageBytes + 8 * kMaxT;   // two input stages, the tables' bounds
    if (per_sm < 0) {
      cudaFuncSetAttribute(k_quantize<D, In, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quantize<D, In, W>, 256, smem) != cudaSuccess ||
          per_sm < 1)
        per_sm = 1;
    }
    unsigned qgrid = (unsigned)((sh.nsm > 0 ? sh.nsm : 152) * per_sm);
    if (qgrid > qsegs) qgrid = qsegs;
    prof_begin(prof, "k_quantize", st);
    launch_k(k_quantize<D, In, W>, qgrid, 256, smem, st, *xmap, sh, ep, w, epoch);
    prof_end(prof, st);

    prof_begin(prof, "k_resolve", st);
    launch_k(k_resolve<D, In, W>, grid, kResolveThreads, 0, st, x, sh, w);
    prof_end(prof, st);
  }
  prof_begin(prof, "k_codebook", st);
  launch_k(k_codebook<W>, sh.U > 0 ? sh.U : 1, 256, 0, st, sh, ep, w, out, cap, out_bytes, chunk_off, epoch);
  prof_end(prof, st);
  if (grid) {
    if (!sh.fold) {
      prof_begin(prof, "k_layout", st);
      launch_k(k_layout<W>, (grid + 7) / 8, 256, 0, st, sh, ep, w, out, cap, out_bytes, chunk_off, epoch);
      prof_end(prof, st);
    }
    prof_begin(prof, "k_emit", st);
    launch_k(k_emit<D, In, W>, grid, kET, emit_stage_bytes<D>(), st, x, sh, w, out, cap, epoch);
    prof_end(prof, st);
  }
}

// Tensor map of x viewed as [B][T][D] (dims innermost first: D, T, B), boxes of
// min(D, 256) elements x 1 table x min(SB, 256) rows; rows past B read as zero.
template <int D, typename In>
static cudaError_t make_x_map(CUtensorMap* map, const In* x, const Shape& sh) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)sh.T, (cuuint64_t)sh.B};
  const cuuint64_t strides[2] = {(cuuint64_t)D * sizeof(In), (cuuint64_t)sh.T * D * sizeof(In)};
  const cuuint32_t box[3] = {(cuuint32_t)QGeo<D, In>::kBoxD, 1u, (cuuint32_t)QGeo<D, In>::kBoxR};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt = sizeof(In) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = encode(map, dt, 3, const_cast<In*>(x), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename In>
static cudaError_t launch_compress_t(const In* x, const Shape& sh, const EbParams& ep, const Work& w, uint8_t* out,
                                    unsigned long long cap, unsigned long long* out_bytes,
                                    unsigned long long* chunk_off, uint32_t epoch, cudaStream_t st, Prof* prof) {
  CUtensorMap xmap;
  if (sh.T > 0 && sh.qseg > 0) {
    cudaError_t e = cudaSuccess;
    switch (sh.D) {
      case 4: e = make_x_map<4, In>(&xmap, x, sh); break;
      case 8: e = make_x_map<8, In>(&xmap, x, sh); break;
      case 16: e = make_x_map<16, In>(&xmap, x, sh); break;
      case 32: e = make_x_map<32, In>(&xmap, x, sh); break;
      case 64: e = make_x_map<64, In>(&xmap, x, sh); break;
      case 128: e = make_x_map<128, In>(&xmap, x, sh); break;
      case 256: e = make_x_map<256, In>(&xmap, x, sh); break;
      case 512: e = make_x_map<512, In>(&xmap, x, sh); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  if (sh.W == 2) {
    switch (sh.D) {
      case 4: launch_compress_d<4, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 8: launch_compress_d<8, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 16: launch_compress_d<16, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 32: launch_compress_d<32, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 64: launch_compress_d<64, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 128: launch_compress_d<128, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 256: launch_compress_d<256, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      case 512: launch_compress_d<512, In, 2>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  switch (sh.D) {
    case 4: launch_compress_d<4, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 8: launch_compress_d<8, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 16: launch_compress_d<16, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 32: launch_compress_d<32, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 64: launch_compress_d<64, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 128: launch_compress_d<128, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 256: launch_compress_d<256, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    case 512: launch_compress_d<512, In, 1>(x, sh, ep, w, out, cap, out_bytes, chunk_off, epoch, st, prof, &xmap); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_compress(const void* x, bool bf16, const Shape& sh, const EbParams& ep, const Work& w,
                            uint8_t* out, unsigned long long cap, unsigned long long* out_bytes,
                            unsigned long long* chunk_off, uint32_t epoch, cudaStream_t st, Prof* prof) {
  return bf16 ? launch_compress_t(static_cast<const uint16_t*>(x), sh, ep, w, out, cap, out_bytes, chunk_off, epoch,
                                  st, prof)
              : launch_compress_t(static_cast<const float*>(x), sh, ep, w, out, cap, out_bytes, chunk_off, epoch,
                                  st, prof);
}

template <int D>
static cudaError_t set_emit_smem() {
  // shared copy of a segment's bitstream: 16 bits per code on average (larger ones go to global memory)
  const cudaError_t e[4] = {
      cudaFuncSetAttribute(k_emit<D, float, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, emit_stage_bytes<D>()),
      cudaFuncSetAttribute(k_emit<D, uint16_t, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, emit_stage_bytes<D>()),
      cudaFuncSetAttribute(k_emit<D, float, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, emit_stage_bytes<D>()),
      cudaFuncSetAttribute(k_emit<D, uint16_t, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, emit_stage_bytes<D>())};
  for (cudaError_t v : e)
    if (v != cudaSuccess) return v;
  return cudaSuccess;
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
