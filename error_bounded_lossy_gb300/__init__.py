"""GB300-native error-bounded lossy compression of DLRM embedding traffic.

Python binding of the C ABI in ``include/ebc.h`` (ctypes; argument marshalling
only).  Every step of compression and decompression runs in the library's
sm_103a CUDA kernels; PyTorch only provides device memory and streams.  There
is no CPU fallback: importing works without a GPU, but every call that needs
the library raises if ``_build/libebc_gb300.so`` is missing.

Method: "Accelerating Communication in Deep Learning Recommendation Model
Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "EBC_OK", "EBC_ERR_INVALID_ARG", "EBC_ERR_CAPACITY", "EBC_ERR_CORRUPT", "EBC_ERR_DEVICE_TIMEOUT",
    "EBC_ERR_CUDA", "EBC_ERR_NO_DEVICE", "EBC_ERR_INTERNAL", "EBC_DECAY_NONE", "EBC_DECAY_LINEAR",
    "EBC_DECAY_STEPWISE", "EBC_DECAY_DROP", "EBC_DECAY_LOG", "EbcStats", "EbcError", "lib", "library_path",
    "ebc_version", "ebc_strerror", "ebc_create", "ebc_destroy", "ebc_set_error_bounds", "ebc_get_error_bounds",
    "ebc_compress_bound", "ebc_compress", "ebc_decompress", "ebc_compress_host", "ebc_decompress_host",
    "ebc_get_stats", "ebc_last_device_error", "ebc_set_profiling", "ebc_get_profile", "Codec",
    "EXPORTED_SYMBOLS", "EbcKernelTime", "EBC_ERR_SCRATCH_LIMIT", "ebc_decompress_noalloc",
    "EBC_MODE_DEDUP_HUFFMAN", "EBC_MODE_HUFFMAN", "EBC_MODE_DEDUP_RAW", "EBC_MODE_RAW", "EbcTableStats",
    "ebc_set_table_modes", "ebc_get_table_stats", "ebc_homo_index", "ebc_speedup", "ebc_select_modes",
    "ebc_select_table_modes", "ebc_table_homo_index", "ebc_set_window", "ebc_compress_bf16",
    "EBC_MAX_CHUNKS", "ebc_compress_chunked_bound", "ebc_compress_chunked", "ebc_compress_chunked_bf16",
    "ebc_decompress_chunked", "EBC_RADIUS", "EBC_RADIUS_WIDE", "ebc_set_radius", "ebc_compress_bound_radius",
    "ebc_decompress_columns", "EbcConfig", "ebc_set_first_wait_polls",
]

EBC_OK, EBC_ERR_INVALID_ARG, EBC_ERR_CAPACITY, EBC_ERR_CORRUPT = 0, 1, 2, 3
EBC_ERR_DEVICE_TIMEOUT, EBC_ERR_CUDA, EBC_ERR_NO_DEVICE, EBC_ERR_INTERNAL = 4, 5, 6, 7
EBC_ERR_SCRATCH_LIMIT = 8
EBC_MAX_CHUNKS = 256
EBC_RADIUS, EBC_RADIUS_WIDE = 128, 512
EBC_MODE_DEDUP_HUFFMAN, EBC_MODE_HUFFMAN, EBC_MODE_DEDUP_RAW, EBC_MODE_RAW = 0, 1, 2, 3
EBC_DECAY_NONE, EBC_DECAY_LINEAR, EBC_DECAY_STEPWISE, EBC_DECAY_DROP, EBC_DECAY_LOG = 0, 1, 2, 3, 4
DECAY = {"none": 0, "linear": 1, "stepwise": 2, "drop": 3, "log": 4}

EXPORTED_SYMBOLS = (
    "ebc_version", "ebc_strerror", "ebc_create", "ebc_destroy", "ebc_set_error_bounds",
    "ebc_get_error_bounds", "ebc_compress_bound", "ebc_compress", "ebc_decompress", "ebc_compress_host",
    "ebc_decompress_host", "ebc_get_stats", "ebc_last_device_error", "ebc_set_profiling", "ebc_get_profile",
    "ebc_decompress_noalloc", "ebc_set_table_modes", "ebc_get_table_stats", "ebc_homo_index", "ebc_speedup",
    "ebc_select_modes", "ebc_select_table_modes", "ebc_table_homo_index", "ebc_set_window", "ebc_compress_bf16",
    "ebc_compress_chunked_bound", "ebc_compress_chunked", "ebc_compress_chunked_bf16", "ebc_decompress_chunked",
    "ebc_set_radius", "ebc_compress_bound_radius", "ebc_decompress_columns", "ebc_set_first_wait_polls",
)


class EbcConfig(ctypes.Structure):
    """ebc_config: options of a context (EbcConfig() is EBC_CONFIG_DEFAULT)."""
    _fields_ = [(n, ctypes.c_int) for n in ("radius", "chunk_vectors", "max_code_len", "dedup", "window")]

    def __init__(self, radius=128, chunk_vectors=0, max_code_len=24, dedup=1, window=0):
        super().__init__(int(radius), int(chunk_vectors), int(max_code_len), int(dedup), int(window))


class EbcStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("in_bytes", "out_bytes", "n_vectors", "n_literal", "n_match",
                                                "n_outlier", "n_chunks", "bitstream_bytes")]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class EbcTableStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("n_literal", "n_match", "n_outlier", "n_chunks", "payload_bits")]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class EbcKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_uint64), ("total_ms", ctypes.c_double)]


class EbcError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {ebc_strerror(code)} ({code})" if what else f"{ebc_strerror(code)} ({code})")


_LOCK = threading.Lock()
_LIB = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded C library; raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"the CUDA library {path} is not built; run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(path)
            P, I, I64, U64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
            sig = {
                "ebc_version": (I, []),
                "ebc_strerror": (ctypes.c_char_p, [I]),
                "ebc_create": (I, [ctypes.POINTER(P), ctypes.POINTER(EbcConfig), I]),
                "ebc_destroy": (None, [P]),
                "ebc_set_error_bounds": (I, [P, P, I, I64, I, D, I64, I]),
                "ebc_get_error_bounds": (I, [P, P, I]),
                "ebc_compress_bound": (U64, [I64, I, I, ctypes.POINTER(EbcConfig)]),
                "ebc_compress": (I, [P, P, I64, I, I, P, P, U64, P, P]),
                "ebc_decompress": (I, [P, P, U64, P, I64, I, I, P]),
                "ebc_compress_host": (I, [P, P, I64, I, I, P, P, U64, P, P]),
                "ebc_decompress_host": (I, [P, P, U64, P, I64, I, I, P]),
                "ebc_get_stats": (I, [P, ctypes.POINTER(EbcStats), P]),
                "ebc_last_device_error": (I, [P]),
                "ebc_set_profiling": (I, [P, I]),
                "ebc_get_profile": (I, [P, ctypes.POINTER(EbcKernelTime), I, ctypes.POINTER(I)]),
                "ebc_decompress_noalloc": (I, [P, U64, P, I64, I, I, P]),
                "ebc_set_table_modes": (I, [P, P, I]),
                "ebc_set_window": (I, [P, I]),
                "ebc_set_first_wait_polls": (I, [P, I]),
                "ebc_compress_bf16": (I, [P, P, I64, I, I, P, P, U64, P, P]),
                "ebc_get_table_stats": (I, [P, ctypes.POINTER(EbcTableStats), I]),
                "ebc_homo_index": (D, [U64, U64]),
                "ebc_speedup": (D, [D, D, D, D]),
                "ebc_select_modes": (I, [P, P, P, D, I, I, P]),
                "ebc_select_table_modes": (I, [P, P, I64, I, I, P, D, P, P]),
                "ebc_table_homo_index": (I, [P, P, I64, I, I, P, P, P]),
                "ebc_compress_chunked_bound": (U64, [I64, I, I, I, I]),
                "ebc_set_radius": (I, [P, I]),
                "ebc_compress_bound_radius": (U64, [I64, I, I, I]),
                "ebc_decompress_columns": (I, [P, P, U64, P, I64, I, I, I, I, P]),
                "ebc_compress_chunked": (I, [P, P, I64, I, I, P, I, P, U64, P, P]),
                "ebc_compress_chunked_bf16": (I, [P, P, I64, I, I, P, I, P, U64, P, P]),
                "ebc_decompress_chunked": (I, [P, P, U64, P, I, P, I64, I, I, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _LIB = L
    return _LIB


# ---- thin wrappers with the C names (plain ints / pointers) ----
def ebc_version() -> int:
    return lib().ebc_version()


def ebc_strerror(code: int) -> str:
    return lib().ebc_strerror(int(code)).decode()


def ebc_create(device: int = 0, config: "EbcConfig | None" = None):
    """A context on `device` with options `config` (None = the defaults)."""
    h = ctypes.c_void_p()
    rc = lib().ebc_create(ctypes.byref(h), ctypes.byref(config) if config is not None else None, int(device))
    if rc:
        raise EbcError(rc, "ebc_create")
    return h


def ebc_destroy(ctx) -> None:
    lib().ebc_destroy(ctx)


def ebc_set_error_bounds(ctx, eb_base_ptr, T, iteration, decay_fn, m0, phase_len, n_steps) -> int:
    return lib().ebc_set_error_bounds(ctx, eb_base_ptr, int(T), int(iteration), int(decay_fn), float(m0),
                                      int(phase_len), int(n_steps))


def ebc_get_error_bounds(ctx, eb_out_ptr, T) -> int:
    return lib().ebc_get_error_bounds(ctx, eb_out_ptr, int(T))


def ebc_compress_bound(B: int, T: int, D: int, config: "EbcConfig | None" = None) -> int:
    return int(lib().ebc_compress_bound(int(B), int(T), int(D),
                                        ctypes.byref(config) if config is not None else None))


def ebc_compress(ctx, d_x, B, T, D, eb_ptr, d_out, out_capacity, d_out_bytes, stream) -> int:
    return lib().ebc_compress(ctx, d_x, int(B), int(T), int(D), eb_ptr, d_out, int(out_capacity), d_out_bytes,
                              stream)


def ebc_decompress(ctx, d_in, in_bytes, d_xhat, B, T, D, stream) -> int:
    return lib().ebc_decompress(ctx, d_in, int(in_bytes), d_xhat, int(B), int(T), int(D), stream)


def ebc_compress_bf16(ctx, d_x, B, T, D, eb_ptr, d_out, out_capacity, d_out_bytes, stream) -> int:
    return lib().ebc_compress_bf16(ctx, d_x, int(B), int(T), int(D), eb_ptr, d_out, int(out_capacity), d_out_bytes,
                                   stream)


def ebc_compress_chunked_bound(B: int, T: int, D: int, n_chunks: int, radius: int = EBC_RADIUS) -> int:
    return int(lib().ebc_compress_chunked_bound(int(B), int(T), int(D), int(n_chunks), int(radius)))


def ebc_set_radius(ctx, radius) -> int:
    return lib().ebc_set_radius(ctx, int(radius))


def ebc_decompress_columns(ctx, d_in, in_bytes, d_xhat, B, T, D, T_out, t_off, stream) -> int:
    return lib().ebc_decompress_columns(ctx, d_in, int(in_bytes), d_xhat, int(B), int(T), int(D), int(T_out),
                                        int(t_off), stream)


def ebc_compress_bound_radius(B: int, T: int, D: int, radius: int) -> int:
    return int(lib().ebc_compress_bound_radius(int(B), int(T), int(D), int(radius)))


def ebc_compress_chunked(ctx, d_x, B, T, D, eb_ptr, n_chunks, d_out, out_capacity, d_offsets, stream) -> int:
    return lib().ebc_compress_chunked(ctx, d_x, int(B), int(T), int(D), eb_ptr, int(n_chunks), d_out,
                                      int(out_capacity), d_offsets, stream)


def ebc_compress_chunked_bf16(ctx, d_x, B, T, D, eb_ptr, n_chunks, d_out, out_capacity, d_offsets, stream) -> int:
    return lib().ebc_compress_chunked_bf16(ctx, d_x, int(B), int(T), int(D), eb_ptr, int(n_chunks), d_out,
                                           int(out_capacity), d_offsets, stream)


def ebc_decompress_chunked(ctx, d_in, in_bytes, d_offsets, n_chunks, d_xhat, B, T, D, stream) -> int:
    return lib().ebc_decompress_chunked(ctx, d_in, int(in_bytes), d_offsets, int(n_chunks), d_xhat, int(B), int(T),
                                        int(D), stream)


def ebc_set_window(ctx, window) -> int:
    return lib().ebc_set_window(ctx, int(window))


def ebc_set_first_wait_polls(ctx, polls) -> int:
    """Test aid: polls of the quantize kernel's first tile wait (negative = the full limit)."""
    return lib().ebc_set_first_wait_polls(ctx, int(polls))


def ebc_set_table_modes(ctx, modes_ptr, T) -> int:
    return lib().ebc_set_table_modes(ctx, modes_ptr, int(T))


def ebc_get_table_stats(ctx, T):
    """(return code, list of EbcTableStats)."""
    arr = (EbcTableStats * max(int(T), 1))()
    rc = lib().ebc_get_table_stats(ctx, arr, int(T))
    return rc, list(arr)[: int(T)]


def ebc_homo_index(n_original, n_compressed) -> float:
    return float(lib().ebc_homo_index(int(n_original), int(n_compressed)))


def ebc_speedup(cr, bw, tc, td) -> float:
    return float(lib().ebc_speedup(float(cr), float(bw), float(tc), float(td)))


def ebc_select_modes(cr_ptr, tc_ptr, td_ptr, bw, T, M, choice_ptr) -> int:
    return lib().ebc_select_modes(cr_ptr, tc_ptr, td_ptr, float(bw), int(T), int(M), choice_ptr)


def ebc_select_table_modes(ctx, d_x, B, T, D, eb_ptr, bw, modes_out_ptr, stream) -> int:
    return lib().ebc_select_table_modes(ctx, d_x, int(B), int(T), int(D), eb_ptr, float(bw), modes_out_ptr, stream)


def ebc_table_homo_index(ctx, d_x, B, T, D, eb_ptr, eta_out_ptr, stream) -> int:
    return lib().ebc_table_homo_index(ctx, d_x, int(B), int(T), int(D), eb_ptr, eta_out_ptr, stream)


def ebc_decompress_noalloc(d_in, in_bytes, d_xhat, B, T, D, stream) -> int:
    """Allocation-free, synchronous decode (no context; static device scratch)."""
    return lib().ebc_decompress_noalloc(d_in, int(in_bytes), d_xhat, int(B), int(T), int(D), stream)


def ebc_compress_host(ctx, h_x, B, T, D, eb_ptr, h_out, out_capacity, out_bytes_ptr, stream) -> int:
    return lib().ebc_compress_host(ctx, h_x, int(B), int(T), int(D), eb_ptr, h_out, int(out_capacity),
                                   out_bytes_ptr, stream)


def ebc_decompress_host(ctx, h_in, in_bytes, h_xhat, B, T, D, stream) -> int:
    return lib().ebc_decompress_host(ctx, h_in, int(in_bytes), h_xhat, int(B), int(T), int(D), stream)


def ebc_get_stats(ctx, stream=None):
    """(return code, EbcStats); stream: a cudaStream_t pointer or None (the last call's)."""
    st = EbcStats()
    rc = lib().ebc_get_stats(ctx, ctypes.byref(st), stream)
    return rc, st


def ebc_last_device_error(ctx) -> int:
    return lib().ebc_last_device_error(ctx)


def ebc_set_profiling(ctx, enable: bool) -> int:
    return lib().ebc_set_profiling(ctx, 1 if enable else 0)


def ebc_get_profile(ctx, capacity: int = 32):
    """{kernel name: (launches, total_ms)} since the last read."""
    arr = (EbcKernelTime * capacity)()
    n = ctypes.c_int(0)
    rc = lib().ebc_get_profile(ctx, arr, capacity, ctypes.byref(n))
    if rc:
        raise EbcError(rc, "ebc_get_profile")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(n.value)}


# ---- torch-facing convenience layer (marshalling only) ----
def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _f32_host(arr, T):
    import numpy as np
    a = np.ascontiguousarray(arr, dtype=np.float32).reshape(-1)
    if a.size != T:
        raise ValueError(f"expected {T} bounds, got {a.size}")
    return a


class Codec:
    """One codec context on one CUDA device.

    compress(x, eb) -> (container uint8 CUDA tensor [capacity], nbytes int64 CUDA tensor [1])
    decompress(container, nbytes_or_len, B, T, D) -> xhat float32 CUDA tensor [B, T, D]
    compress_chunked(x, n, eb) -> (buffer, offsets [n + 1]): one container per batch slice
    decompress_chunked(buffer, nbytes, offsets, B, T, D) -> xhat
    decompress_columns(container, nbytes, T, out, t_off): a sender's tables into columns of out
    set_window(w), set_table_modes(modes), set_radius(128 | 512): options of later calls
    """

    def __init__(self, device: int = 0, config: "EbcConfig | None" = None):
        import torch
        self.device = torch.device("cuda", device)
        self._ctx = ebc_create(device, config)
        self.radius = config.radius if config is not None and config.radius else EBC_RADIUS

    def close(self):
        if self._ctx is not None:
            ebc_destroy(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._ctx

    def set_error_bounds(self, eb_base, iteration: int, fn="stepwise", m0: float = 2.0, phase_len: int = 0,
                         n_steps: int = 1):
        import numpy as np
        a = np.ascontiguousarray(eb_base, dtype=np.float32).reshape(-1)
        fn = DECAY[fn] if isinstance(fn, str) else int(fn)
        rc = ebc_set_error_bounds(self._ctx, a.ctypes.data_as(ctypes.c_void_p), a.size, iteration, fn, m0,
                                  phase_len, n_steps)
        if rc:
            raise EbcError(rc, "ebc_set_error_bounds")

    def error_bounds(self, T: int):
        import numpy as np
        out = np.zeros(T, np.float32)
        rc = ebc_get_error_bounds(self._ctx, out.ctypes.data_as(ctypes.c_void_p), T)
        if rc:
            raise EbcError(rc, "ebc_get_error_bounds")
        return out

    def compress_bound(self, B, T, D) -> int:
        """Worst-case container bytes with this context's alphabet."""
        return ebc_compress_bound_radius(B, T, D, self.radius)

    def set_radius(self, radius: int) -> None:
        """Alphabet of later calls: 128 (8-bit codes) or 512 (the wide alphabet)."""
        rc = ebc_set_radius(self._ctx, radius)
        if rc:
            raise EbcError(rc, "ebc_set_radius")
        self.radius = int(radius)

    def compress_into(self, x, eb, out, nbytes, stream=None) -> None:
        """Asynchronous compress of CUDA tensor x [B,T,D] into preallocated out / nbytes."""
        import torch
        B, T, D = x.shape
        ebh = None if eb is None else _f32_host(eb, T)
        fn, name = (ebc_compress_bf16, "ebc_compress_bf16") if x.dtype == torch.bfloat16 else (ebc_compress,
                                                                                               "ebc_compress")
        rc = fn(self._ctx, _ptr(x), B, T, D, ebh.ctypes.data_as(ctypes.c_void_p) if ebh is not None else None,
                _ptr(out), out.numel(), _ptr(nbytes), _stream_ptr(stream))
        if rc:
            raise EbcError(rc, name)

    def compress(self, x, eb=None, stream=None, out=None):
        import torch
        if not (x.is_cuda and x.dtype in (torch.float32, torch.bfloat16) and x.is_contiguous() and x.dim() == 3):
            raise ValueError("x must be a contiguous float32 or bfloat16 CUDA tensor [B, T, D]")
        B, T, D = x.shape
        cap = self.compress_bound(B, T, D)
        if out is None:
            out = torch.empty(max(cap, 16), dtype=torch.uint8, device=x.device)
        nbytes = torch.zeros(1, dtype=torch.int64, device=x.device)
        self.compress_into(x, eb, out, nbytes, stream)
        return out, nbytes

    def compress_chunked_bound(self, B, T, D, n_chunks) -> int:
        return ebc_compress_chunked_bound(B, T, D, n_chunks, self.radius)

    def compress_chunked(self, x, n_chunks: int, eb=None, stream=None, out=None, offsets=None):
        """One container per slice of the batch (numpy array_split slices), back to
        back in one buffer.  Returns (buffer uint8, offsets int64 [n_chunks + 1]),
        both CUDA tensors; container r spans [offsets[r], offsets[r+1])."""
        import torch
        if not (x.is_cuda and x.dtype in (torch.float32, torch.bfloat16) and x.is_contiguous() and x.dim() == 3):
            raise ValueError("x must be a contiguous float32 or bfloat16 CUDA tensor [B, T, D]")
        B, T, D = x.shape
        if out is None:
            out = torch.empty(max(self.compress_chunked_bound(B, T, D, n_chunks), 16), dtype=torch.uint8,
                              device=x.device)
        if offsets is None:
            offsets = torch.zeros(n_chunks + 1, dtype=torch.int64, device=x.device)
        ebh = None if eb is None else _f32_host(eb, T)
        fn, name = ((ebc_compress_chunked_bf16, "ebc_compress_chunked_bf16") if x.dtype == torch.bfloat16
                    else (ebc_compress_chunked, "ebc_compress_chunked"))
        rc = fn(self._ctx, _ptr(x), B, T, D, ebh.ctypes.data_as(ctypes.c_void_p) if ebh is not None else None,
                n_chunks, _ptr(out), out.numel(), _ptr(offsets), _stream_ptr(stream))
        if rc:
            raise EbcError(rc, name)
        return out, offsets

    def decompress_chunked(self, buf, in_bytes: int, offsets, B: int, T: int, D: int, stream=None, out=None):
        """Restores every slice of the batch from its container (offsets: CUDA int64 [n + 1])."""
        import torch
        if out is None:
            out = torch.empty((B, T, D), dtype=torch.float32, device=buf.device)
        rc = ebc_decompress_chunked(self._ctx, _ptr(buf), in_bytes, _ptr(offsets), offsets.numel() - 1, _ptr(out),
                                    B, T, D, _stream_ptr(stream))
        if rc:
            raise EbcError(rc, "ebc_decompress_chunked")
        return out

    def decompress_columns(self, container, in_bytes: int, T: int, out, t_off: int, stream=None):
        """Restores a container of T tables into columns [t_off, t_off + T) of out
        (CUDA float32 [B, T_out, D]); the other columns are not touched."""
        B, T_out, D = out.shape
        rc = ebc_decompress_columns(self._ctx, _ptr(container), in_bytes, _ptr(out), B, T, D, T_out, t_off,
                                    _stream_ptr(stream))
        if rc:
            raise EbcError(rc, "ebc_decompress_columns")
        return out

    def decompress_into(self, container, in_bytes: int, xhat, stream=None) -> None:
        B, T, D = xhat.shape
        rc = ebc_decompress(self._ctx, _ptr(container), in_bytes, _ptr(xhat), B, T, D, _stream_ptr(stream))
        if rc:
            raise EbcError(rc, "ebc_decompress")

    def decompress(self, container, in_bytes: int, B: int, T: int, D: int, stream=None, out=None):
        import torch
        if out is None:
            out = torch.empty((B, T, D), dtype=torch.float32, device=container.device)
        self.decompress_into(container, in_bytes, out, stream)
        return out

    def set_profiling(self, enable: bool) -> None:
        rc = ebc_set_profiling(self._ctx, enable)
        if rc:
            raise EbcError(rc, "ebc_set_profiling")

    def profile(self) -> dict:
        return ebc_get_profile(self._ctx)

    def last_error(self) -> int:
        return ebc_last_device_error(self._ctx)

    def check(self) -> None:
        rc = self.last_error()
        if rc:
            raise EbcError(rc, "device")

    def set_window(self, window: int) -> None:
        """Dedup window in rows for the following compress calls (0 = whole batch)."""
        rc = ebc_set_window(self._ctx, window)
        if rc:
            raise EbcError(rc, "ebc_set_window")

    def set_table_modes(self, modes) -> None:
        """Per-table modes (0..3) for the following compress calls; None restores mode 0."""
        import numpy as np
        if modes is None:
            rc = ebc_set_table_modes(self._ctx, None, 0)
        else:
            a = np.ascontiguousarray(modes, dtype=np.uint8).reshape(-1)
            rc = ebc_set_table_modes(self._ctx, a.ctypes.data_as(ctypes.c_void_p), a.size)
        if rc:
            raise EbcError(rc, "ebc_set_table_modes")

    def table_stats(self, T: int) -> list:
        rc, st = ebc_get_table_stats(self._ctx, T)
        if rc:
            raise EbcError(rc, "ebc_get_table_stats")
        return [s.as_dict() for s in st]

    def select_table_modes(self, x, eb, bandwidth: float, stream=None):
        """Eq. (2) per-table mode choice measured on the sample batch x (CUDA [B, T, D])."""
        import numpy as np
        B, T, D = x.shape
        e = np.ascontiguousarray(eb, dtype=np.float32).reshape(-1)
        out = np.zeros(T, dtype=np.uint8)
        rc = ebc_select_table_modes(self._ctx, ctypes.c_void_p(x.data_ptr()), B, T, D,
                                    e.ctypes.data_as(ctypes.c_void_p), bandwidth,
                                    out.ctypes.data_as(ctypes.c_void_p), _stream_ptr(stream))
        if rc:
            raise EbcError(rc, "ebc_select_table_modes")
        return out

    def table_homo_index(self, x, eb, stream=None):
        """Eq. (1) Homogenization Index of each table of the batch x (CUDA [B, T, D])."""
        import numpy as np
        B, T, D = x.shape
        e = np.ascontiguousarray(eb, dtype=np.float32).reshape(-1)
        out = np.zeros(T, dtype=np.float64)
        rc = ebc_table_homo_index(self._ctx, ctypes.c_void_p(x.data_ptr()), B, T, D,
                                  e.ctypes.data_as(ctypes.c_void_p), out.ctypes.data_as(ctypes.c_void_p),
                                  _stream_ptr(stream))
        if rc:
            raise EbcError(rc, "ebc_table_homo_index")
        return out

    def stats(self) -> dict:
        rc, st = ebc_get_stats(self._ctx)
        d = st.as_dict()
        d["device_error"] = rc
        return d

    def compress_host(self, x_host, eb=None, out_host=None):
        """Synchronous compress of a host float32 array/tensor (pinned is fastest)."""
        import numpy as np
        import torch
        xt = x_host if isinstance(x_host, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x_host))
        B, T, D = xt.shape
        ebh = None if eb is None else _f32_host(eb, T)
        cap = self.compress_bound(B, T, D)
        if out_host is None:
            out_host = torch.empty(max(cap, 16), dtype=torch.uint8)
        n = ctypes.c_uint64(0)
        rc = ebc_compress_host(self._ctx, ctypes.c_void_p(xt.data_ptr()), B, T, D,
                               ebh.ctypes.data_as(ctypes.c_void_p) if ebh is not None else None,
                               ctypes.c_void_p(out_host.data_ptr()), out_host.numel(), ctypes.byref(n),
                               _stream_ptr(None))
        if rc:
            raise EbcError(rc, "ebc_compress_host")
        return out_host, int(n.value)

    def decompress_host(self, container_host, in_bytes: int, B: int, T: int, D: int, out_host=None):
        import torch
        if out_host is None:
            out_host = torch.empty((B, T, D), dtype=torch.float32)
        rc = ebc_decompress_host(self._ctx, ctypes.c_void_p(container_host.data_ptr()), in_bytes,
                                 ctypes.c_void_p(out_host.data_ptr()), B, T, D, _stream_ptr(None))
        if rc:
            raise EbcError(rc, "ebc_decompress_host")
        return out_host
