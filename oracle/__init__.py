"""CPU oracle of the error-bounded embedding codec (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg are the only importers.  The product library
never imports, links or executes anything here, and the oracle shares no code
with it: ``ebc_oracle.c`` re-implements the container format from its
specification.

Method: "Accelerating Communication in Deep Learning Recommendation Model
Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
sections III-C (error-bound schedule), III-D (quantization encoder,
vector-based LZ, Huffman) and III-E (single-buffer layout).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ebc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libebc_oracle.so")
_LOCK = threading.Lock()
_LIB = None

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3
DECAY = {"none": 0, "linear": 1, "stepwise": 2, "drop": 3, "log": 4}
LMAX = 24
RADIUS = 128
RADIUS_WIDE = 512   # the wide alphabet: 1024 symbols, 16-bit codes


class Info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("n_literal", "n_match", "n_outlier", "n_chunks", "bitstream_bytes", "total_bytes")]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction); returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            P, I64, U64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
            lib.ebo_quantize.argtypes = [P, I64, ctypes.c_float, P]
            lib.ebo_quantize.restype = I64
            lib.ebo_dequantize.argtypes = [I, ctypes.c_float]
            lib.ebo_dequantize.restype = ctypes.c_float
            lib.ebo_vector_hash.argtypes = [P, P, I]
            lib.ebo_vector_hash.restype = ctypes.c_uint32
            lib.ebo_huffman_lengths.argtypes = [P, I, P]
            lib.ebo_huffman_lengths.restype = I
            lib.ebo_canonical_codes.argtypes = [P, I, P]
            lib.ebo_canonical_codes.restype = I
            lib.ebo_decay_factor.argtypes = [I, I64, ctypes.c_double, I64, I]
            lib.ebo_decay_factor.restype = ctypes.c_double
            lib.ebo_compress_bound.argtypes = [I64, I, I]
            lib.ebo_compress_bound.restype = U64
            lib.ebo_compress.argtypes = [P, I64, I, I, P, P, U64, ctypes.POINTER(Info), P, P, P]
            lib.ebo_compress.restype = I
            lib.ebo_decompress.argtypes = [P, U64, I64, I, I, P, P]
            lib.ebo_decompress.restype = I
            lib.ebo_compress_modes.argtypes = [P, I64, I, I, P, P, P, U64, ctypes.POINTER(Info), P, P, P]
            lib.ebo_compress_modes.restype = I
            lib.ebo_compress_ex.argtypes = [P, I64, I, I, P, P, I, P, U64, ctypes.POINTER(Info), P, P, P]
            lib.ebo_compress_ex.restype = I
            lib.ebo_homo_index.argtypes = [U64, U64]
            lib.ebo_homo_index.restype = ctypes.c_double
            lib.ebo_speedup.argtypes = [ctypes.c_double] * 4
            lib.ebo_speedup.restype = ctypes.c_double
            lib.ebo_select_modes.argtypes = [P, P, P, ctypes.c_double, I, I, P]
            lib.ebo_select_modes.restype = I
            lib.ebo_quantize_r.argtypes = [P, I64, ctypes.c_float, I, P]
            lib.ebo_quantize_r.restype = I64
            lib.ebo_dequantize_r.argtypes = [I, ctypes.c_float, I]
            lib.ebo_dequantize_r.restype = ctypes.c_float
            lib.ebo_vector_hash_r.argtypes = [P, P, I, I]
            lib.ebo_vector_hash_r.restype = ctypes.c_uint32
            lib.ebo_huffman_lengths_n.argtypes = [P, I, I, P]
            lib.ebo_huffman_lengths_n.restype = I
            lib.ebo_canonical_codes_n.argtypes = [P, I, I, P]
            lib.ebo_canonical_codes_n.restype = I
            lib.ebo_compress_bound_r.argtypes = [I64, I, I, I]
            lib.ebo_compress_bound_r.restype = U64
            lib.ebo_compress_r.argtypes = [P, I64, I, I, P, P, I, I, P, U64, ctypes.POINTER(Info), P, P, P]
            lib.ebo_compress_r.restype = I
            lib.ebo_decompress_r.argtypes = [P, U64, I64, I, I, P, P]
            lib.ebo_decompress_r.restype = I
            _LIB = lib
    return _LIB


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def quantize(x, eb: float) -> np.ndarray:
    """Quantization codes (uint8; 0 = outlier) of a float32 array under bound eb."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    sym = np.empty(x.shape, dtype=np.uint8)
    r = _lib().ebo_quantize(_ptr(x), x.size, float(eb), _ptr(sym))
    if r < 0:
        raise ValueError("invalid error bound")
    return sym


def dequantize(sym: int, eb: float, radius: int = RADIUS) -> float:
    return float(_lib().ebo_dequantize_r(int(sym), float(eb), int(radius)))


def quantize_r(x, eb: float, radius: int) -> np.ndarray:
    """Quantization codes (uint16; 0 = outlier, else q + radius) with radius 128 or 512."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    sym = np.empty(x.shape, dtype=np.uint16)
    r = _lib().ebo_quantize_r(_ptr(x), x.size, float(eb), int(radius), _ptr(sym))
    if r < 0:
        raise ValueError("invalid error bound or radius")
    return sym


def vector_hash(sym_row, x_row, radius: int = RADIUS) -> int:
    x = np.ascontiguousarray(x_row, dtype=np.float32)
    if radius == RADIUS:
        s = np.ascontiguousarray(sym_row, dtype=np.uint8)
        return int(_lib().ebo_vector_hash(_ptr(s), _ptr(x), s.size))
    s = np.ascontiguousarray(sym_row, dtype=np.uint16)
    return int(_lib().ebo_vector_hash_r(_ptr(s), _ptr(x), s.size, int(radius)))


def huffman_lengths(freq, lmax: int = LMAX, symbols: int = 256):
    """(lengths uint8[symbols], halving rounds) of the two-queue Huffman code
    over an alphabet of 256 or 1024 symbols."""
    f = np.zeros(symbols, dtype=np.uint64)
    freq = np.asarray(freq, dtype=np.uint64)
    f[: freq.size] = freq
    ln = np.zeros(symbols, dtype=np.uint8)
    if symbols == 256:
        rounds = _lib().ebo_huffman_lengths(_ptr(f), int(lmax), _ptr(ln))
    else:
        rounds = _lib().ebo_huffman_lengths_n(_ptr(f), int(symbols), int(lmax), _ptr(ln))
    if rounds < 0:
        raise ValueError("bad arguments")
    return ln, rounds


def canonical_codes(lens, lmax: int = LMAX) -> np.ndarray:
    ln = np.ascontiguousarray(lens, dtype=np.uint8)
    code = np.zeros(ln.size, dtype=np.uint32)
    if _lib().ebo_canonical_codes_n(_ptr(ln), ln.size, int(lmax), _ptr(code)) < 0:
        raise ValueError("lengths violate the Kraft inequality")
    return code


def decay_factor(fn, iteration: int, m0: float, phase_len: int, n_steps: int = 1) -> float:
    fn = DECAY[fn] if isinstance(fn, str) else int(fn)
    return float(_lib().ebo_decay_factor(fn, int(iteration), float(m0), int(phase_len), int(n_steps)))


def scheduled_bounds(eb_base, fn, iteration, m0, phase_len, n_steps=1) -> np.ndarray:
    """eb_t(i) = fl32(base_t * factor(i)), factor in double."""
    f = decay_factor(fn, iteration, m0, phase_len, n_steps)
    base = np.asarray(eb_base, dtype=np.float32).astype(np.float64)
    return (base * f).astype(np.float32)


def compress_bound(B: int, T: int, D: int, radius: int = RADIUS) -> int:
    return int(_lib().ebo_compress_bound_r(int(B), int(T), int(D), int(radius)))


MODE_DEDUP_HUFFMAN, MODE_HUFFMAN, MODE_DEDUP_RAW, MODE_RAW = 0, 1, 2, 3


def compress(x, eb, *, want_internals: bool = False, modes=None, window: int = 0, radius: int = RADIUS):
    """Compress x [B,T,D] float32 with per-table bounds eb [T] and, optionally,
    per-table modes [T] (0 dedup + Huffman, 1 Huffman only, 2 dedup + raw
    codes, 3 raw codes only), a dedup window (0 = whole batch, first
    occurrence; 1..255 = nearest earlier vector within that many rows) and the
    quantization radius (128, or 512 for the wide 1024-symbol alphabet).

    Returns (container uint8 array, info dict) and, with want_internals,
    also (sym [T,B,D] uint8 (uint16 with radius 512), ref [T,B] uint32,
    lens [T, 2 * radius] uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    B, T, D = x.shape
    eb = np.ascontiguousarray(eb, dtype=np.float32)
    assert eb.shape == (T,)
    cap = compress_bound(B, T, D, radius)
    if cap == 0 and B * T * D > 0:
        raise ValueError("unsupported shape")
    out = np.zeros(max(cap, 16), dtype=np.uint8)
    info = Info()
    sym = np.empty((T, B, D), dtype=np.uint16) if want_internals else None
    ref = np.empty((T, B), dtype=np.uint32) if want_internals else None
    lens = np.empty((T, 2 * radius), dtype=np.uint8) if want_internals else None
    md = None
    if modes is not None:
        md = np.ascontiguousarray(modes, dtype=np.uint8)
        assert md.shape == (T,)
    rc = _lib().ebo_compress_r(_ptr(x), B, T, D, _ptr(eb), _ptr(md) if md is not None else None, int(window),
                               int(radius), _ptr(out), out.size, ctypes.byref(info),
                                   _ptr(sym) if sym is not None else None,
                                   _ptr(ref) if ref is not None else None,
                                   _ptr(lens) if lens is not None else None)
    if rc != OK:
        raise RuntimeError(f"oracle compress failed: {rc}")
    d = {k: int(getattr(info, k)) for k, _ in Info._fields_}
    buf = out[: d["total_bytes"]].copy()
    if want_internals:
        return buf, d, (sym.astype(np.uint8) if radius == RADIUS else sym), ref, lens
    return buf, d


def decompress_rc(buf, B: int, T: int, D: int):
    """(return code, xhat [B,T,D], sym [T,B,D]) without raising; sym is uint8,
    or uint16 for a container of the wide alphabet (radius field 512)."""
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    xhat = np.zeros((B, T, D), dtype=np.float32)
    wide = buf.size >= 28 and int.from_bytes(bytes(buf[24:28]), "little") == RADIUS_WIDE
    sym = np.zeros((T, B, D), dtype=np.uint16)
    rc = _lib().ebo_decompress_r(_ptr(buf), buf.size, int(B), int(T), int(D), _ptr(xhat), _ptr(sym))
    return rc, xhat, (sym if wide else sym.astype(np.uint8))


def decompress(buf, B: int, T: int, D: int):
    rc, xhat, sym = decompress_rc(buf, B, T, D)
    if rc != OK:
        raise RuntimeError(f"oracle decompress failed: {rc}")
    return xhat, sym


def homo_index(n_original: int, n_compressed: int) -> float:
    """Eq. (1) Homogenization Index of one table."""
    return float(_lib().ebo_homo_index(int(n_original), int(n_compressed)))


def speedup(cr: float, bw: float, tc: float, td: float) -> float:
    """Eq. (2) theoretical speed-up."""
    return float(_lib().ebo_speedup(float(cr), float(bw), float(tc), float(td)))


def select_modes(cr, tc, td, bw: float):
    """Per-table argmax of Eq. (2) over M candidates: cr [T, M], tc [M], td [M]."""
    cr = np.ascontiguousarray(cr, dtype=np.float64)
    T, M = cr.shape
    tc = np.ascontiguousarray(tc, dtype=np.float64)
    td = np.ascontiguousarray(td, dtype=np.float64)
    out = np.zeros(T, dtype=np.uint8)
    rc = _lib().ebo_select_modes(_ptr(cr), _ptr(tc), _ptr(td), float(bw), T, M, _ptr(out))
    if rc != OK:
        raise ValueError("bad selection arguments")
    return out


def chunk_rows(B: int, n_chunks: int):
    """Row ranges [b0, b1) of the n_chunks slices of a batch of B rows.

    §III-E "Buffer Optimization" and §IV-D: the batch is split equally into
    one slice per destination rank of the all-to-all.  Where B is not a
    multiple of n_chunks, the first B % n_chunks slices take one row more
    (slices past B are empty)."""
    if n_chunks < 1:
        raise ValueError("n_chunks must be >= 1")
    q, rem = divmod(int(B), int(n_chunks))
    starts = [r * q + min(r, rem) for r in range(n_chunks + 1)]
    return [(starts[r], starts[r + 1]) for r in range(n_chunks)]


def compress_chunked(x, eb, n_chunks: int, *, modes=None, window: int = 0, radius: int = RADIUS):
    """§III-E "Buffer Optimization", Fig. 7 (top): every slice of the batch is
    compressed on its own, as a self-contained container, and the containers
    lie back to back in one sending buffer.  Returns (buffer uint8, offsets
    uint64 [n_chunks + 1]): container r spans [offsets[r], offsets[r+1])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    B = x.shape[0]
    parts, offs = [], [0]
    for b0, b1 in chunk_rows(B, n_chunks):
        buf, _ = compress(x[b0:b1], eb, modes=modes, window=window, radius=radius)
        parts.append(buf)
        offs.append(offs[-1] + buf.size)
    return np.concatenate(parts), np.asarray(offs, dtype=np.uint64)


def decompress_chunked(buf, offsets, B: int, T: int, D: int):
    """Fig. 7 (bottom): container r of the buffer restores rows
    chunk_rows(B, n)[r] of the batch, independently of the others."""
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    offsets = [int(v) for v in offsets]
    xhat = np.zeros((B, T, D), dtype=np.float32)
    for r, (b0, b1) in enumerate(chunk_rows(B, len(offsets) - 1)):
        xh, _ = decompress(buf[offsets[r]:offsets[r + 1]], b1 - b0, T, D)
        xhat[b0:b1] = xh
    return xhat


def decompress_columns(buf, B: int, T: int, D: int, T_out: int, t_off: int, out=None):
    """The receiving side of the all-to-all (§III-E, Fig. 7 bottom): a container
    of T tables restores columns [t_off, t_off + T) of an output [B, T_out, D];
    the other columns are left as they are."""
    if not (0 <= t_off and t_off + T <= T_out):
        raise ValueError("columns out of range")
    if out is None:
        out = np.zeros((B, T_out, D), dtype=np.float32)
    xh, _ = decompress(buf, B, T, D)
    out[:, t_off:t_off + T] = xh
    return out
