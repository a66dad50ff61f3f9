// ebc_api.cu -- host side of the C ABI declared in include/ebc.h: argument
// checks, the error-bound schedule, device scratch, and the kernel launches.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "ebc_internal.cuh"


using namespace ebc;

// Per-kernel timing: a pool of CUDA event pairs recorded around each launch
// while profiling is on; read back (and cleared) by ebc_get_profile.
struct ebc::Prof {
  static constexpr int kPairs = 8192;
  cudaEvent_t ev[2 * kPairs] = {};
  const char* name[kPairs] = {};
  int used = 0;
  bool on = false;
  bool created = false;
};

void ebc::prof_begin(Prof* p, const char* name, cudaStream_t st) {
  if (!p || !p->on || p->used >= Prof::kPairs) return;
  p->name[p->used] = name;
  cudaEventRecord(p->ev[2 * p->used], st);
}

void ebc::prof_end(Prof* p, cudaStream_t st) {
  if (!p || !p->on || p->used >= Prof::kPairs) return;
  cudaEventRecord(p->ev[2 * p->used + 1], st);
  ++p->used;
}

struct ebc_ctx {
  int device = 0;
  cudaStream_t last_stream = nullptr;
  Glob* glob = nullptr;                // device
  unsigned long long* h_pinned = nullptr;  // pinned scratch for the host-buffer calls
  // compress scratch
  void* cbuf = nullptr;
  size_t cbuf_bytes = 0;
  // decompress scratch
  void* dbuf = nullptr;
  size_t dbuf_bytes = 0;
  const void* dclean_buf = nullptr;    // dbuf whose decoder accumulators, dclean_bytes long, are zero
  size_t dclean_bytes = 0;
  // host-buffer staging
  void* stage_in = nullptr;
  size_t stage_in_bytes = 0;
  void* stage_out = nullptr;
  size_t stage_out_bytes = 0;
  unsigned long long* d_nbytes = nullptr;
  uint32_t cepoch = 0, depoch = 0;
  int nsm = 0;
  // the compress layout whose dedup table and look-back flags are known clean
  const void* clean_buf = nullptr;
  int64_t cleanB = -1;
  int cleanT = -1, cleanD = -1, cleanR = -1, cleanW = -1;
  // schedule
  float* eb_base = nullptr;
  float* eb_now = nullptr;
  int sched_T = 0;
  // per-table coding modes (0 = dedup + Huffman for every table when modes_T == 0)
  int window = 0;                      // dedup window of the compress calls (0 = whole batch)
  int radius = kRadius;                // alphabet of the compress and decompress calls (128 or 512)
  uint32_t mode_or = 0;                // modes added to every table's (kModeNoDedup: dedup off by config)
  int first_wait = kWaitLimit;         // polls of the quantize kernel's first tile wait (test aid)
  uint8_t* d_modes = nullptr;          // device [kMaxT]
  uint8_t h_modes[kMaxT] = {};
  int modes_T = 0;
  // last compress shape
  int64_t lastB = 0;
  int lastT = 0, lastD = 0, lastR = 1, lastRadius = kRadius;
  Prof* prof = nullptr;
};

// ---------------------------------------------------------------------------
// shapes and argument checks
// ---------------------------------------------------------------------------
static bool dim_ok(int D) { return D >= 4 && D <= 512 && (D & (D - 1)) == 0; }

static bool shape_ok(int64_t B, int T, int D) {
  if (B < 0 || B > kMaxB || T < 0 || T > kMaxT || !dim_ok(D)) return false;
  return (uint64_t)B * (uint64_t)T * (uint64_t)D <= (1ull << 31);
}

// R: slices of the batch, each coded as a container of its own (1 = one container).
// radius: 128 (8-bit codes) or 512 (the wide alphabet, 16-bit codes).
static Shape make_shape(int64_t B, int T, int D, int nsm = 0, int window = 0, int R = 1, int radius = kRadius) {
  Shape sh;
  sh.W = radius == kRadiusWide ? 2 : 1;
  sh.A = 2 * radius;
  sh.T_out = T;
  sh.t_off = 0;
  sh.first_wait = kWaitLimit;
  sh.nsm = nsm;
  sh.B = B;
  sh.T = T;
  sh.D = D;
  sh.R = R;
  sh.U = R * T;
  sh.Bq = B / R;
  sh.Brem = (int)(B % R);
  sh.Bc = sh.Bq + (sh.Brem > 0 ? 1 : 0);
  sh.SB = 8192 / D < 32 ? 32 : 8192 / D;
  sh.KC = 128 / D < 1 ? 1 : 128 / D;
  sh.qseg = (int)((B + sh.SB - 1) / sh.SB);
  sh.nseg = (int)((sh.Bc + sh.SB - 1) / sh.SB);
  sh.nw = (int)((sh.Bc + 31) / 32);
  uint32_t S = 64;
  while ((int64_t)S < 2 * sh.Bc) S <<= 1;
  sh.S = S;
  sh.window = window;
  sh.ref_bytes = window > 0 ? 1 : (B <= 65536 ? 2 : 4);
  sh.symstride = ((uint64_t)B * (uint64_t)D * (uint64_t)sh.W + 15u) & ~(uint64_t)15u;
  // per-unit segment offsets inside k_codebook for short units of the 8-bit alphabet; otherwise (long
  // units, or 1024-bin histograms) k_layout spreads that work over all SMs
  sh.fold = sh.nseg <= kFoldMaxSeg && sh.W == 1 ? 1 : 0;
  return sh;
}

static uint64_t pad16h(uint64_t n) { return (n + 15u) & ~(uint64_t)15u; }

// Bytes of the container that do not depend on the data: header, table and
// segment records, match bitmap.
static uint64_t fixed_bytes(const Shape& sh) {
  return kHeaderBytes + (uint64_t)sh.T * table_rec_bytes(sh.A) + (uint64_t)sh.T * sh.nseg * kSegRecBytes +
         pad16h((uint64_t)sh.T * sh.nw * 4u);
}

static bool eb_ok(float eb) {
  if (!(eb >= 1.17549435e-38f) || !(eb <= 3.40282347e+38f)) return false;
  const volatile float ebx2 = 2.0f * eb;
  if (!(ebx2 <= 3.40282347e+38f)) return false;
  const volatile float inv = 1.0f / ebx2;
  return inv >= 1.17549435e-38f;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static int cuda_err(cudaError_t e) { return e == cudaSuccess ? EBC_OK : EBC_ERR_CUDA; }

// ---------------------------------------------------------------------------
// scratch
// ---------------------------------------------------------------------------
namespace {
struct Carver {
  char* base;
  size_t off = 0;
  template <class P>
  P* take(size_t bytes) {
    P* p = reinterpret_cast<P*>(base ? base + off : nullptr);
    off += (bytes + 255) & ~(size_t)255;
    return p;
  }
};
}  // namespace

static Work carve_compress(void* buf, const Shape& sh, Glob* g, size_t* total) {
  Carver c{reinterpret_cast<char*>(buf)};
  Work w{};
  const size_t nvec = (size_t)sh.B * sh.T, nsegT = (size_t)sh.U * sh.nseg, U = (size_t)sh.U;
  w.slots = c.take<unsigned long long>(8 * U * sh.S);
  const size_t groups = (nsegT + 7) / 8 > U ? (nsegT + 7) / 8 : U;
  w.seg_desc = c.take<uint4>(16 * groups);
  w.tile_base = c.take<uint4>(16 * groups);
  w.seg_base = c.take<uint4>(16 * nsegT);
  w.sym = c.take<uint8_t>((size_t)sh.T * sh.symstride);
  w.vhash = c.take<uint32_t>(4 * nvec);
  w.ref = c.take<uint32_t>(4 * nvec);
  w.bitmap = c.take<uint32_t>(4 * U * sh.nw);
  w.seg_hist = c.take<uint32_t>(4 * (size_t)sh.A * nsegT);
  w.seg_cnt = c.take<uint4>(16 * nsegT);
  w.tab_hist = c.take<uint32_t>(4 * (size_t)sh.A * U);
  w.tab_cnt = c.take<uint4>(16 * U);
  w.tab_rec = c.take<uint4>(16 * U);
  w.tab_bits = c.take<unsigned long long>(8 * U);
  w.modes = nullptr;
  w.tabcode = c.take<uint32_t>(4 * (size_t)sh.A * U);
  w.cont = c.take<ContLay>(sizeof(ContLay) * (size_t)sh.R);
  w.glob = g;
  *total = c.off;
  return w;
}

// The accumulators come first, so that their bytes (which must be zero before
// a call) are the same for every shape with as many units and containers.
static Work carve_decompress(void* buf, const Shape& sh, Glob* g, size_t* total, size_t* acc_bytes = nullptr) {
  Carver c{reinterpret_cast<char*>(buf)};
  Work w{};
  w.uacc = c.take<uint4>(16 * (size_t)(sh.U > 0 ? sh.U : 1));
  w.cacc = c.take<uint2>(8 * (size_t)sh.R);
  if (acc_bytes) *acc_bytes = c.off;
  w.lay = c.take<Layout>(sizeof(Layout) * (size_t)sh.R);
  w.srcrow = c.take<uint32_t>(4 * (size_t)sh.B * (size_t)sh.T);
  w.glob = g;
  *total = c.off;
  return w;
}

static int grow(void** buf, size_t* have, size_t need) {
  if (need <= *have && *buf) return EBC_OK;
  if (*buf) {
    if (cudaDeviceSynchronize() != cudaSuccess) return EBC_ERR_CUDA;
    cudaFree(*buf);
    *buf = nullptr;
    *have = 0;
  }
  if (need == 0) need = 256;
  if (cudaMalloc(buf, need) != cudaSuccess) {
    *buf = nullptr;
    return EBC_ERR_CUDA;
  }
  *have = need;
  return EBC_OK;
}

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

int ebc_version(void) { return EBC_VERSION; }

const char* ebc_strerror(int code) {
  switch (code) {
    case EBC_OK: return "ok";
    case EBC_ERR_INVALID_ARG: return "invalid argument";
    case EBC_ERR_CAPACITY: return "output buffer too small for the container";
    case EBC_ERR_CORRUPT: return "corrupt container";
    case EBC_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case EBC_ERR_CUDA: return "CUDA runtime error";
    case EBC_ERR_NO_DEVICE: return "no usable sm_103 device";
    case EBC_ERR_INTERNAL: return "internal invariant failed on the device";
    case EBC_ERR_SCRATCH_LIMIT: return "shape needs more than the 16 MiB static scratch of ebc_decompress_noalloc";
    default: return "unknown error";
  }
}

// A config the format can honour: the radius is 128 or 512, the chunk size and
// the longest code are the format's own (0 selects them), dedup is on or off,
// the window is 0..255.
static bool config_ok(const ebc_config* cfg) {
  if (!cfg) return true;
  const bool radius = cfg->radius == 0 || cfg->radius == kRadius || cfg->radius == kRadiusWide;
  return radius && cfg->chunk_vectors == 0 && (cfg->max_code_len == 0 || cfg->max_code_len == kLmax) &&
         (cfg->dedup == 0 || cfg->dedup == 1) && cfg->window >= 0 && cfg->window <= kMaxWindow;
}

static int config_radius(const ebc_config* cfg) { return cfg && cfg->radius ? cfg->radius : kRadius; }

int ebc_create(ebc_ctx** out, const ebc_config* cfg, int device) {
  if (!out) return EBC_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg)) return EBC_ERR_INVALID_ARG;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return EBC_ERR_NO_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return EBC_ERR_NO_DEVICE;
  if (!(prop.major == 10 && prop.minor == 3)) return EBC_ERR_NO_DEVICE;
  if (cudaSetDevice(device) != cudaSuccess) return EBC_ERR_CUDA;
  ebc_ctx* c = new (std::nothrow) ebc_ctx();
  if (!c) return EBC_ERR_INTERNAL;
  c->device = device;
  c->nsm = prop.multiProcessorCount;
  c->radius = config_radius(cfg);
  c->window = cfg ? cfg->window : 0;
  c->mode_or = cfg && cfg->dedup == 0 ? kModeNoDedup : 0u;
  if (cudaMalloc(&c->glob, sizeof(Glob)) != cudaSuccess || cudaMemset(c->glob, 0, sizeof(Glob)) != cudaSuccess ||
      cudaMalloc(&c->d_nbytes, 16) != cudaSuccess || cudaMallocHost(&c->h_pinned, 64) != cudaSuccess ||
      cudaMalloc(&c->d_modes, kMaxT) != cudaSuccess) {
    ebc_destroy(c);
    return EBC_ERR_CUDA;
  }
  if (set_kernel_attributes() != cudaSuccess || set_decoder_attributes() != cudaSuccess) {
    ebc_destroy(c);
    return EBC_ERR_CUDA;
  }
  *out = c;
  return EBC_OK;
}

void ebc_destroy(ebc_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  cudaFree(c->glob);
  cudaFree(c->cbuf);
  cudaFree(c->dbuf);
  cudaFree(c->stage_in);
  cudaFree(c->stage_out);
  cudaFree(c->d_nbytes);
  cudaFree(c->d_modes);
  if (c->h_pinned) cudaFreeHost(c->h_pinned);
  std::free(c->eb_base);
  std::free(c->eb_now);
  if (c->prof) {
    if (c->prof->created)
      for (cudaEvent_t e : c->prof->ev) cudaEventDestroy(e);
    delete c->prof;
  }
  delete c;
}

// The decay factor and the scheduled bound are computed in double and rounded
// once to float; the same expressions, in the same order, define the schedule
// in the header.
static double decay_factor(int fn, int64_t i, double m0, int64_t P, int S) {
  if (fn == EBC_DECAY_NONE || P <= 0 || i >= P) return 1.0;
  if (i < 0) i = 0;
  const double frac = (double)i / (double)P;
  switch (fn) {
    case EBC_DECAY_LINEAR: return m0 - (m0 - 1.0) * frac;
    case EBC_DECAY_STEPWISE: {
      if (S < 1) S = 1;
      const int64_t k = (i * (int64_t)S) / P;
      return m0 - (m0 - 1.0) * ((double)k / (double)S);
    }
    case EBC_DECAY_DROP: return m0;
    case EBC_DECAY_LOG: return std::pow(m0, 1.0 - frac);
    default: return 1.0;
  }
}

int ebc_set_error_bounds(ebc_ctx* c, const float* eb_base, int T, int64_t iteration, int decay_fn, double m0,
                         int64_t phase_len, int n_steps) {
  if (!c || !eb_base || T < 1 || T > kMaxT || decay_fn < EBC_DECAY_NONE || decay_fn > EBC_DECAY_LOG ||
      iteration < 0 || !(m0 > 0.0) || !std::isfinite(m0) || (decay_fn == EBC_DECAY_STEPWISE && n_steps < 1))
    return EBC_ERR_INVALID_ARG;
  const double f = decay_factor(decay_fn, iteration, m0, phase_len, n_steps);
  float* base = (float*)std::malloc(sizeof(float) * T);
  float* now = (float*)std::malloc(sizeof(float) * T);
  if (!base || !now) {
    std::free(base);
    std::free(now);
    return EBC_ERR_INTERNAL;
  }
  for (int t = 0; t < T; ++t) {
    base[t] = eb_base[t];
    now[t] = (float)((double)eb_base[t] * f);
    if (!eb_ok(base[t]) || !eb_ok(now[t])) {
      std::free(base);
      std::free(now);
      return EBC_ERR_INVALID_ARG;
    }
  }
  std::free(c->eb_base);
  std::free(c->eb_now);
  c->eb_base = base;
  c->eb_now = now;
  c->sched_T = T;
  return EBC_OK;
}

int ebc_get_error_bounds(const ebc_ctx* c, float* eb_out, int T) {
  if (!c || !eb_out || T != c->sched_T || !c->eb_now) return EBC_ERR_INVALID_ARG;
  std::memcpy(eb_out, c->eb_now, sizeof(float) * T);
  return EBC_OK;
}

static bool radius_ok(int radius) { return radius == kRadius || radius == kRadiusWide; }

uint64_t ebc_compress_bound(int64_t B, int T, int D, const ebc_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return ebc_compress_bound_radius(B, T, D, config_radius(cfg));
}

uint64_t ebc_compress_bound_radius(int64_t B, int T, int D, int radius) {
  if (!shape_ok(B, T, D) || !radius_ok(radius)) return 0;
  const Shape sh = make_shape(B, T, D, 0, 0, 1, radius);
  const uint64_t N = (uint64_t)B * T * D, nvec = (uint64_t)B * T;
  const uint64_t words = (N * (kLmax + 32) + 31) / 32 + 4ull * T * sh.nseg;
  return fixed_bytes(sh) + pad16h(nvec * 2u) + pad16h(nvec * sh.ref_bytes) + words * 4u;
}

// Sum of the data-independent bytes of the containers of R slices.
static uint64_t fixed_bytes_sliced(int64_t B, int T, int D, int R, int radius) {
  const Shape all = make_shape(B, T, D, 0, 0, R);
  uint64_t n = 0;
  for (int r = 0; r < R; ++r) n += fixed_bytes(make_shape(slice_rows(all, r), T, D, 0, 0, 1, radius));
  return n;
}

uint64_t ebc_compress_chunked_bound(int64_t B, int T, int D, int n_chunks, int radius) {
  if (!shape_ok(B, T, D) || n_chunks < 1 || n_chunks > kMaxSlices || !radius_ok(radius)) return 0;
  const Shape all = make_shape(B, T, D, 0, 0, n_chunks);
  uint64_t n = 0;
  for (int r = 0; r < n_chunks; ++r) n += ebc_compress_bound_radius(slice_rows(all, r), T, D, radius);
  return n;
}

// fp32 or bf16 input (bf16: its raw 16 bits; compressed as its exact fp32 value), in R slices
// (d_offsets: null for one container, else [R + 1] container boundaries written on the device)
static int compress_any(ebc_ctx* c, const void* d_x, bool bf16, int64_t B, int T, int D, const float* eb, int R,
                        void* d_out, uint64_t out_capacity, uint64_t* d_out_bytes, uint64_t* d_offsets,
                        void* stream) {
  if (!c || !shape_ok(B, T, D) || R < 1 || R > kMaxSlices || !d_out || !d_out_bytes || !aligned16(d_out) ||
      ((uintptr_t)d_out_bytes & 7u) != 0 || (bf16 && D < 8))
    return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && (!d_x || !aligned16(d_x))) return EBC_ERR_INVALID_ARG;
  if (c->modes_T != 0 && c->modes_T != T) return EBC_ERR_INVALID_ARG;
  const float* ebs = eb;
  if (!ebs) {
    if (!c->eb_now || c->sched_T != T) return EBC_ERR_INVALID_ARG;
    ebs = c->eb_now;
  }
  EbParams ep;
  std::memset(&ep, 0, sizeof ep);
  for (int t = 0; t < T; ++t) {
    if (!eb_ok(ebs[t])) return EBC_ERR_INVALID_ARG;
    ep.eb[t] = ebs[t];
  }
  Shape sh = make_shape(B, T, D, c->nsm, c->window, R, c->radius);
  sh.first_wait = c->first_wait;
  if (out_capacity < (R == 1 ? fixed_bytes(sh) : fixed_bytes_sliced(B, T, D, R, c->radius))) return EBC_ERR_CAPACITY;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  size_t need = 0;
  carve_compress(nullptr, sh, c->glob, &need);
  int rc = grow(&c->cbuf, &c->cbuf_bytes, need);
  if (rc) return rc;
  Work w = carve_compress(c->cbuf, sh, c->glob, &need);
  w.modes = c->modes_T ? c->d_modes : nullptr;
  w.mode_or = c->mode_or;
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  c->cepoch = (c->cepoch + 1) & 0xFFFFFFu;
  c->lastB = B;
  c->lastT = T;
  c->lastD = D;
  c->lastR = R;
  c->lastRadius = c->radius;
  // Each call leaves its dedup table empty (k_emit).  A new layout on this
  // buffer starts from a reset.
  if (T > 0 && sh.nseg > 0 &&
      (c->clean_buf != c->cbuf || c->cleanB != B || c->cleanT != T || c->cleanD != D || c->cleanR != R ||
       c->cleanW != sh.W)) {
    if (cudaMemsetAsync(w.slots, 0xFF, 8 * (size_t)sh.U * sh.S, st) != cudaSuccess) return EBC_ERR_CUDA;
    c->clean_buf = c->cbuf;
    c->cleanB = B;
    c->cleanT = T;
    c->cleanD = D;
    c->cleanR = R;
    c->cleanW = sh.W;
  }
  const cudaError_t e = launch_compress(d_x, bf16, sh, ep, w, (uint8_t*)d_out, out_capacity,
                                        (unsigned long long*)d_out_bytes, (unsigned long long*)d_offsets,
                                        c->cepoch, st, c->prof);
  if (e != cudaSuccess) c->clean_buf = nullptr;   // the dedup table may be left dirty
  return cuda_err(e);
}

int ebc_compress(ebc_ctx* c, const float* d_x, int64_t B, int T, int D, const float* eb, void* d_out,
                 uint64_t out_capacity, uint64_t* d_out_bytes, void* stream) {
  return compress_any(c, d_x, false, B, T, D, eb, 1, d_out, out_capacity, d_out_bytes, nullptr, stream);
}

int ebc_compress_bf16(ebc_ctx* c, const uint16_t* d_x, int64_t B, int T, int D, const float* eb, void* d_out,
                      uint64_t out_capacity, uint64_t* d_out_bytes, void* stream) {
  return compress_any(c, d_x, true, B, T, D, eb, 1, d_out, out_capacity, d_out_bytes, nullptr, stream);
}

int ebc_compress_chunked(ebc_ctx* c, const float* d_x, int64_t B, int T, int D, const float* eb, int n_chunks,
                         void* d_out, uint64_t out_capacity, uint64_t* d_offsets, void* stream) {
  if (!d_offsets || n_chunks < 1 || n_chunks > kMaxSlices) return EBC_ERR_INVALID_ARG;
  return compress_any(c, d_x, false, B, T, D, eb, n_chunks, d_out, out_capacity, d_offsets + n_chunks, d_offsets,
                      stream);
}

int ebc_compress_chunked_bf16(ebc_ctx* c, const uint16_t* d_x, int64_t B, int T, int D, const float* eb,
                              int n_chunks, void* d_out, uint64_t out_capacity, uint64_t* d_offsets, void* stream) {
  if (!d_offsets || n_chunks < 1 || n_chunks > kMaxSlices) return EBC_ERR_INVALID_ARG;
  return compress_any(c, d_x, true, B, T, D, eb, n_chunks, d_out, out_capacity, d_offsets + n_chunks, d_offsets,
                      stream);
}

// T_out, t_off: the output rows hold T_out tables and the container's tables go to columns
// [t_off, t_off + T) (T_out = T, t_off = 0 for a whole batch)
static int decompress_any(ebc_ctx* c, const void* d_in, uint64_t in_bytes, const uint64_t* d_offsets, int R,
                          float* d_xhat, int64_t B, int T, int D, void* stream, int T_out = -1, int t_off = 0) {
  Shape sh = make_shape(B, T, D, c->nsm, 0, R, c->radius);
  if (T_out >= 0) {
    sh.T_out = T_out;
    sh.t_off = t_off;
  }
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  size_t need = 0, acc = 0;
  carve_decompress(nullptr, sh, c->glob, &need);
  int rc = grow(&c->dbuf, &c->dbuf_bytes, need);
  if (rc) return rc;
  const Work w = carve_decompress(c->dbuf, sh, c->glob, &need, &acc);
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  c->depoch = (c->depoch + 1) & 0xFFFFFFu;
  // The decoder's accumulators are left zero by every call.  A call whose
  // accumulators span other bytes than the last call's (where a windowed call's
  // row-source table may have been written since) clears them first.
  if (c->dclean_buf != c->dbuf || c->dclean_bytes != acc) {
    if (cudaMemsetAsync(c->dbuf, 0, acc, st) != cudaSuccess) return EBC_ERR_CUDA;
    c->dclean_buf = c->dbuf;
    c->dclean_bytes = acc;
  }
  const cudaError_t e = launch_decompress((const uint8_t*)d_in, in_bytes, (const unsigned long long*)d_offsets, sh,
                                          w, d_xhat, c->depoch, st, c->prof);
  if (e != cudaSuccess) c->dclean_buf = nullptr;   // the accumulators may be left dirty
  return cuda_err(e);
}

int ebc_decompress(ebc_ctx* c, const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B, int T, int D,
                   void* stream) {
  if (!c || !shape_ok(B, T, D) || !d_in || !aligned16(d_in)) return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && (!d_xhat || !aligned16(d_xhat))) return EBC_ERR_INVALID_ARG;
  return decompress_any(c, d_in, in_bytes, nullptr, 1, d_xhat, B, T, D, stream);
}

int ebc_decompress_columns(ebc_ctx* c, const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B, int T, int D,
                           int T_out, int t_off, void* stream) {
  if (!c || !shape_ok(B, T, D) || !shape_ok(B, T_out, D) || t_off < 0 || (int64_t)t_off + T > T_out || !d_in ||
      !aligned16(d_in))
    return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T_out * D;
  if (N > 0 && (!d_xhat || !aligned16(d_xhat))) return EBC_ERR_INVALID_ARG;
  return decompress_any(c, d_in, in_bytes, nullptr, 1, d_xhat, B, T, D, stream, T_out, t_off);
}

int ebc_decompress_chunked(ebc_ctx* c, const void* d_in, uint64_t in_bytes, const uint64_t* d_offsets,
                           int n_chunks, float* d_xhat, int64_t B, int T, int D, void* stream) {
  if (!c || !shape_ok(B, T, D) || !d_in || !aligned16(d_in) || !d_offsets || ((uintptr_t)d_offsets & 7u) != 0 ||
      n_chunks < 1 || n_chunks > kMaxSlices)
    return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && (!d_xhat || !aligned16(d_xhat))) return EBC_ERR_INVALID_ARG;
  return decompress_any(c, d_in, in_bytes, d_offsets, n_chunks, d_xhat, B, T, D, stream);
}

int ebc_set_radius(ebc_ctx* c, int radius) {
  if (!c || !radius_ok(radius)) return EBC_ERR_INVALID_ARG;
  c->radius = radius;
  return EBC_OK;
}

int ebc_set_first_wait_polls(ebc_ctx* c, int polls) {
  if (!c || polls > kWaitLimit) return EBC_ERR_INVALID_ARG;
  c->first_wait = polls < 0 ? kWaitLimit : polls;
  return EBC_OK;
}

int ebc_set_window(ebc_ctx* c, int window) {
  if (!c || window < 0 || window > kMaxWindow) return EBC_ERR_INVALID_ARG;
  c->window = window;
  return EBC_OK;
}

int ebc_set_table_modes(ebc_ctx* c, const uint8_t* modes, int T) {
  if (!c) return EBC_ERR_INVALID_ARG;
  if (!modes || T == 0) {
    c->modes_T = 0;
    return EBC_OK;
  }
  if (T < 0 || T > kMaxT) return EBC_ERR_INVALID_ARG;
  for (int t = 0; t < T; ++t)
    if (modes[t] > (kModeNoDedup | kModeRawCodes)) return EBC_ERR_INVALID_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  // no call of this context may still be reading the previous modes
  if (cudaDeviceSynchronize() != cudaSuccess) return EBC_ERR_CUDA;
  if (cudaMemcpy(c->d_modes, modes, (size_t)T, cudaMemcpyHostToDevice) != cudaSuccess) return EBC_ERR_CUDA;
  std::memcpy(c->h_modes, modes, (size_t)T);
  c->modes_T = T;
  return EBC_OK;
}

int ebc_get_table_stats(ebc_ctx* c, ebc_table_stats* out, int T) {
  if (!c || !out || T <= 0 || T != c->lastT) return EBC_ERR_INVALID_ARG;
  const int err = ebc_last_device_error(c);
  if (err == EBC_ERR_CUDA) return err;
  const Shape sh = make_shape(c->lastB, T, c->lastD, c->nsm, c->window, c->lastR, c->lastRadius);
  std::memset(out, 0, sizeof(*out) * (size_t)T);
  if (sh.nseg == 0 || !c->cbuf) return err;   // an empty batch: nothing was coded
  size_t need = 0;
  const Work w = carve_compress(c->cbuf, sh, c->glob, &need);   // the last compress's layout
  const size_t U = (size_t)sh.U;
  uint4* cnt = new (std::nothrow) uint4[U];
  unsigned long long* bits = new (std::nothrow) unsigned long long[U];
  int rc = err;
  if (!cnt || !bits) {
    rc = EBC_ERR_INTERNAL;
  } else if (cudaMemcpy(cnt, w.tab_cnt, 16 * U, cudaMemcpyDeviceToHost) != cudaSuccess ||
             cudaMemcpy(bits, w.tab_bits, 8 * U, cudaMemcpyDeviceToHost) != cudaSuccess) {
    rc = EBC_ERR_CUDA;
  } else {
    for (size_t u = 0; u < U; ++u) {   // a table's counts over all slices
      const int t = (int)(u % (size_t)T);
      out[t].n_literal += cnt[u].x;
      out[t].n_match += cnt[u].y;
      out[t].n_outlier += cnt[u].z;
      out[t].n_chunks += cnt[u].w;
      out[t].payload_bits += bits[u];
    }
  }
  delete[] cnt;
  delete[] bits;
  return rc;
}

double ebc_homo_index(uint64_t n_original, uint64_t n_compressed) {
  if (n_original == 0) return 0.0;
  return ((double)n_original - (double)n_compressed) / (double)n_original;
}

double ebc_speedup(double cr, double bw, double tc, double td) {
  if (!(cr > 0.0) || !(tc > 0.0) || !(td > 0.0) || bw < 0.0) return 0.0;
  return 1.0 / (1.0 / cr + bw * (1.0 / tc + 1.0 / td));
}

int ebc_select_modes(const double* cr, const double* tc, const double* td, double bw, int T, int M,
                     uint8_t* choice) {
  if (T < 0 || M < 1 || M > 255 || (T > 0 && (!cr || !tc || !td || !choice))) return EBC_ERR_INVALID_ARG;
  for (int t = 0; t < T; ++t) {
    int best = 0;
    double top = ebc_speedup(cr[(size_t)t * M], bw, tc[0], td[0]);
    for (int m = 1; m < M; ++m) {
      const double s = ebc_speedup(cr[(size_t)t * M + m], bw, tc[m], td[m]);
      if (s > top) {
        top = s;
        best = m;
      }
    }
    choice[t] = (uint8_t)best;
  }
  return EBC_OK;
}

int ebc_last_device_error(ebc_ctx* c) {
  if (!c) return EBC_ERR_INVALID_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  if (cudaStreamSynchronize(c->last_stream) != cudaSuccess) return EBC_ERR_CUDA;
  unsigned int code = 0;
  if (cudaMemcpy(&code, &c->glob->sticky, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return EBC_ERR_CUDA;
  if (code) {
    const unsigned int zero = 0;
    if (cudaMemcpy(&c->glob->sticky, &zero, 4, cudaMemcpyHostToDevice) != cudaSuccess) return EBC_ERR_CUDA;
  }
  return (int)code;
}

int ebc_get_stats(ebc_ctx* c, ebc_stats* out, void* stream) {
  if (!c || !out) return EBC_ERR_INVALID_ARG;
  const int err = ebc_last_device_error(c);   // the last call has completed
  if (err == EBC_ERR_CUDA) return err;
  cudaStream_t st = stream ? (cudaStream_t)stream : c->last_stream;
  Glob g;
  if (cudaMemcpyAsync(&g, c->glob, sizeof g, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return EBC_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  out->n_vectors = (uint64_t)c->lastB * c->lastT;
  out->in_bytes = out->n_vectors * c->lastD * 4u;
  out->out_bytes = g.total;
  out->n_literal = g.n_lit;
  out->n_match = g.n_match;
  out->n_outlier = g.n_out;
  out->n_chunks = g.n_chunks;
  out->bitstream_bytes = g.words * 4u;
  return err;
}

int ebc_compress_host(ebc_ctx* c, const float* h_x, int64_t B, int T, int D, const float* eb, void* h_out,
                      uint64_t out_capacity, uint64_t* out_bytes, void* stream) {
  if (!c || !shape_ok(B, T, D) || !h_out || !out_bytes) return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && !h_x) return EBC_ERR_INVALID_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  const uint64_t bound = ebc_compress_bound_radius(B, T, D, c->radius);
  int rc = grow(&c->stage_in, &c->stage_in_bytes, N * 4u);
  if (!rc) rc = grow(&c->stage_out, &c->stage_out_bytes, bound);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (N > 0 && cudaMemcpyAsync(c->stage_in, h_x, N * 4u, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return EBC_ERR_CUDA;
  rc = ebc_compress(c, (const float*)c->stage_in, B, T, D, eb, c->stage_out, bound, (uint64_t*)c->d_nbytes, stream);
  if (rc) return rc;
  if (cudaMemcpyAsync(c->h_pinned, c->d_nbytes, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return EBC_ERR_CUDA;
  const int err = ebc_last_device_error(c);
  if (err) return err;
  const uint64_t n = c->h_pinned[0];
  *out_bytes = n;
  if (n > out_capacity) return EBC_ERR_CAPACITY;
  if (cudaMemcpyAsync(h_out, c->stage_out, n, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return EBC_ERR_CUDA;
  return EBC_OK;
}

int ebc_decompress_host(ebc_ctx* c, const void* h_in, uint64_t in_bytes, float* h_xhat, int64_t B, int T, int D,
                        void* stream) {
  if (!c || !shape_ok(B, T, D) || !h_in) return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && !h_xhat) return EBC_ERR_INVALID_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  int rc = grow(&c->stage_out, &c->stage_out_bytes, in_bytes);
  if (!rc) rc = grow(&c->stage_in, &c->stage_in_bytes, N * 4u);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (in_bytes && cudaMemcpyAsync(c->stage_out, h_in, in_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return EBC_ERR_CUDA;
  rc = ebc_decompress(c, c->stage_out, in_bytes, (float*)c->stage_in, B, T, D, stream);
  if (rc) return rc;
  if (N > 0 && cudaMemcpyAsync(h_xhat, c->stage_in, N * 4u, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return EBC_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return EBC_ERR_CUDA;
  return ebc_last_device_error(c);
}

int ebc_set_profiling(ebc_ctx* c, int enable) {
  if (!c) return EBC_ERR_INVALID_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return EBC_ERR_CUDA;
  if (!c->prof) {
    c->prof = new (std::nothrow) Prof();
    if (!c->prof) return EBC_ERR_INTERNAL;
  }
  if (enable && !c->prof->created) {
    for (cudaEvent_t& e : c->prof->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return EBC_ERR_CUDA;
    c->prof->created = true;
  }
  c->prof->on = enable != 0;
  return EBC_OK;
}

int ebc_get_profile(ebc_ctx* c, ebc_kernel_time* out, int capacity, int* count) {
  if (!c || !count || capacity < 0 || (capacity > 0 && !out)) return EBC_ERR_INVALID_ARG;
  *count = 0;
  if (!c->prof || !c->prof->created) return EBC_OK;
  Prof* p = c->prof;
  if (p->used > 0 && cudaEventSynchronize(p->ev[2 * p->used - 1]) != cudaSuccess) return EBC_ERR_CUDA;
  int n = 0;
  for (int i = 0; i < p->used; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p->ev[2 * i], p->ev[2 * i + 1]) != cudaSuccess) return EBC_ERR_CUDA;
    int k = 0;
    while (k < n && std::strncmp(out[k].name, p->name[i], sizeof out[k].name) != 0) ++k;
    if (k == n) {
      if (n == capacity) continue;
      std::memset(&out[k], 0, sizeof out[k]);
      std::strncpy(out[k].name, p->name[i], sizeof out[k].name - 1);
      ++n;
    }
    out[k].launches += 1;
    out[k].total_ms += ms;
  }
  p->used = 0;
  *count = n;
  return EBC_OK;
}


// Compresses (and, with d_xhat, decompresses) one batch in the given mode for
// every table; returns the per-table stats and the event-timed durations.
static int run_mode(ebc_ctx* c, const float* d_x, int64_t B, int T, int D, const float* eb, int mode,
                    ebc_table_stats* stats, float* ms_c, float* ms_d, cudaStream_t st) {
  uint8_t modes[kMaxT];
  std::memset(modes, mode, (size_t)T);
  int rc = ebc_set_table_modes(c, modes, T);
  if (rc) return rc;
  const uint64_t N = (uint64_t)B * T * D;
  const uint64_t cap = ebc_compress_bound_radius(B, T, D, c->radius);
  rc = grow(&c->stage_out, &c->stage_out_bytes, cap);
  if (!rc) rc = grow(&c->stage_in, &c->stage_in_bytes, N * 4u);
  if (rc) return rc;
  cudaEvent_t ev[4];
  for (cudaEvent_t& e : ev)
    if (cudaEventCreate(&e) != cudaSuccess) return EBC_ERR_CUDA;
  // a warm-up call, then a timed one of each direction
  rc = ebc_compress(c, d_x, B, T, D, eb, c->stage_out, cap, (uint64_t*)c->d_nbytes, st);
  if (!rc && cudaEventRecord(ev[0], st) != cudaSuccess) rc = EBC_ERR_CUDA;
  if (!rc) rc = ebc_compress(c, d_x, B, T, D, eb, c->stage_out, cap, (uint64_t*)c->d_nbytes, st);
  if (!rc && (cudaEventRecord(ev[1], st) != cudaSuccess ||
              cudaMemcpyAsync(c->h_pinned, c->d_nbytes, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
              cudaStreamSynchronize(st) != cudaSuccess))
    rc = EBC_ERR_CUDA;
  if (!rc) rc = ebc_get_table_stats(c, stats, T);
  const uint64_t n = c->h_pinned[0];
  if (!rc) rc = ebc_decompress(c, c->stage_out, n, (float*)c->stage_in, B, T, D, st);
  if (!rc && cudaEventRecord(ev[2], st) != cudaSuccess) rc = EBC_ERR_CUDA;
  if (!rc) rc = ebc_decompress(c, c->stage_out, n, (float*)c->stage_in, B, T, D, st);
  if (!rc && (cudaEventRecord(ev[3], st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)) rc = EBC_ERR_CUDA;
  if (!rc) rc = ebc_last_device_error(c);
  if (!rc && (cudaEventElapsedTime(ms_c, ev[0], ev[1]) != cudaSuccess ||
              cudaEventElapsedTime(ms_d, ev[2], ev[3]) != cudaSuccess))
    rc = EBC_ERR_CUDA;
  for (cudaEvent_t& e : ev) cudaEventDestroy(e);
  return rc;
}

// Restores the caller's modes (and the context's dedup switch, which the
// sampling runs turn back on) after a sampling run.
static int restore_modes(ebc_ctx* c, int saved_T, const uint8_t* saved, uint32_t saved_or) {
  c->mode_or = saved_or;
  return ebc_set_table_modes(c, saved_T ? saved : nullptr, saved_T);
}

int ebc_select_table_modes(ebc_ctx* c, const float* d_x, int64_t B, int T, int D, const float* eb, double bw,
                           uint8_t* modes_out, void* stream) {
  if (!c || !shape_ok(B, T, D) || T == 0 || B == 0 || !eb || !modes_out || !d_x || bw < 0.0)
    return EBC_ERR_INVALID_ARG;
  const int saved_T = c->modes_T;
  uint8_t saved[kMaxT];
  std::memcpy(saved, c->h_modes, (size_t)kMaxT);
  const uint32_t saved_or = c->mode_or;
  c->mode_or = 0;   // every candidate mode as such
  const Shape sh = make_shape(B, T, D, c->nsm, c->window, 1, c->radius);
  const double raw_bytes = 4.0 * (double)B * D;   // per table
  const double fixed = (double)table_rec_bytes(sh.A) + (double)kSegRecBytes * sh.nseg + 4.0 * sh.nw;
  double* cr = new (std::nothrow) double[(size_t)T * 4];
  ebc_table_stats* st = new (std::nothrow) ebc_table_stats[(size_t)T];
  double tc[4], td[4];
  int rc = (!cr || !st) ? EBC_ERR_INTERNAL : EBC_OK;
  for (int m = 0; m < 4 && !rc; ++m) {
    float ms_c = 0.f, ms_d = 0.f;
    rc = run_mode(c, d_x, B, T, D, eb, m, st, &ms_c, &ms_d, (cudaStream_t)stream);
    if (rc) break;
    tc[m] = raw_bytes * T / (ms_c * 1e-3);
    td[m] = raw_bytes * T / (ms_d * 1e-3);
    for (int t = 0; t < T; ++t) {
      const double bytes = (double)st[t].payload_bits / 8.0 + 2.0 * st[t].n_chunks +
                           (double)sh.ref_bytes * st[t].n_match + fixed;
      cr[(size_t)t * 4 + m] = raw_bytes / bytes;
    }
  }
  const int rr = restore_modes(c, saved_T, saved, saved_or);
  if (!rc) rc = rr;
  if (!rc) rc = ebc_select_modes(cr, tc, td, bw, T, 4, modes_out);
  delete[] cr;
  delete[] st;
  return rc;
}

int ebc_table_homo_index(ebc_ctx* c, const float* d_x, int64_t B, int T, int D, const float* eb,
                         double* eta_out, void* stream) {
  if (!c || !shape_ok(B, T, D) || T == 0 || !eb || !eta_out || (B > 0 && !d_x)) return EBC_ERR_INVALID_ARG;
  const int saved_T = c->modes_T;
  uint8_t saved[kMaxT];
  std::memcpy(saved, c->h_modes, (size_t)kMaxT);
  const uint32_t saved_or = c->mode_or;
  c->mode_or = 0;   // N_compressed counts distinct quantized vectors: dedup on
  float* tiny = new (std::nothrow) float[(size_t)T];
  ebc_table_stats* a = new (std::nothrow) ebc_table_stats[(size_t)T];
  ebc_table_stats* b = new (std::nothrow) ebc_table_stats[(size_t)T];
  int rc = (!tiny || !a || !b) ? EBC_ERR_INTERNAL : EBC_OK;
  if (!rc) {
    for (int t = 0; t < T; ++t) tiny[t] = 1.17549435e-38f;   // the smallest admissible bound
    rc = ebc_set_table_modes(c, nullptr, 0);
  }
  const uint64_t cap = ebc_compress_bound_radius(B, T, D, c->radius);
  if (!rc) rc = grow(&c->stage_out, &c->stage_out_bytes, cap);
  cudaStream_t s = (cudaStream_t)stream;
  if (!rc) rc = ebc_compress(c, d_x, B, T, D, eb, c->stage_out, cap, (uint64_t*)c->d_nbytes, s);
  if (!rc) rc = ebc_get_table_stats(c, a, T);
  if (!rc) rc = ebc_compress(c, d_x, B, T, D, tiny, c->stage_out, cap, (uint64_t*)c->d_nbytes, s);
  if (!rc) rc = ebc_get_table_stats(c, b, T);
  if (!rc)
    for (int t = 0; t < T; ++t) eta_out[t] = ebc_homo_index(b[t].n_literal, a[t].n_literal);
  const int rr = restore_modes(c, saved_T, saved, saved_or);
  if (!rc) rc = rr;
  delete[] tiny;
  delete[] a;
  delete[] b;
  return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decompression
//
// Some callers cannot allocate device memory when they decode: a process whose
// device memory has been handed to another allocator (a framework's caching
// pool) gets an out-of-memory error or fragmentation from cudaMalloc, and in a
// latency-bound loop cudaMalloc/cudaFree synchronise the device and stall the
// other streams.  ebc_decompress_noalloc serves them: it runs the same decoder
// kernels as ebc_decompress, but their scratch (status block, decode tables,
// chunk descriptors, literal-row and match lists) is carved from the static
// device array below instead of a context's buffer.
// ---------------------------------------------------------------------------

// The array is part of this library's device image: every GPU on which the
// image is loaded holds these 16 MiB until the process exits.  Its first 256
// bytes hold the status block (Glob); the decoder's tables follow.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
constexpr size_t kNoAllocGlobBytes = 256;
static_assert(sizeof(Glob) <= kNoAllocGlobBytes, "status block does not fit its slot");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int nsm = 0;
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device, with that device current: check it is an sm_103 part and
// look up the device address of the scratch array.  (On the host the array's
// name is only a stand-in symbol, never a pointer a kernel may be given.)
int noalloc_setup(int dev, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, nsm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return EBC_ERR_NO_DEVICE;
    if (!(major == 10 && minor == 3)) return EBC_ERR_NO_DEVICE;
    if (set_decoder_attributes() != cudaSuccess) return EBC_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return EBC_ERR_CUDA;
    d.scratch = static_cast<unsigned char*>(p);
    d.nsm = nsm;
    d.ready = true;
  }
  *out = &d;
  return EBC_OK;
}
}  // namespace

extern "C" {

int ebc_decompress_noalloc(const void* d_in, uint64_t in_bytes, float* d_xhat, int64_t B, int T, int D,
                           void* stream) {
  if (!shape_ok(B, T, D) || !d_in || !aligned16(d_in)) return EBC_ERR_INVALID_ARG;
  const uint64_t N = (uint64_t)B * T * D;
  if (N > 0 && (!d_xhat || !aligned16(d_xhat))) return EBC_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return EBC_ERR_NO_DEVICE;
  NoAllocDevice* nd = nullptr;
  int rc = noalloc_setup(dev, &nd);
  if (rc) return rc;
  const Shape sh = make_shape(B, T, D, nd->nsm);
  size_t need = 0, acc = 0;
  carve_decompress(nullptr, sh, nullptr, &need);
  if (need > kNoAllocScratchBytes - kNoAllocGlobBytes) return EBC_ERR_SCRATCH_LIMIT;
  Glob* g = reinterpret_cast<Glob*>(nd->scratch);
  const Work w = carve_decompress(nd->scratch + kNoAllocGlobBytes, sh, g, &need, &acc);
  cudaStream_t st = (cudaStream_t)stream;
  // The array keeps whatever the previous call left; the status block and the
  // decoder's count accumulators must start at zero (everything else is
  // written before it is read).
  if (cudaMemsetAsync(g, 0, kNoAllocGlobBytes + acc, st) != cudaSuccess) return EBC_ERR_CUDA;
  if (launch_decompress((const uint8_t*)d_in, in_bytes, nullptr, sh, w, d_xhat, 1u, st, nullptr) != cudaSuccess)
    return EBC_ERR_CUDA;
  unsigned int code = 0;
  if (cudaMemcpyAsync(&code, &g->sticky, sizeof code, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return EBC_ERR_CUDA;
  return (int)code;
}

}  // extern "C"
