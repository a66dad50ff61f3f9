"""Seeded synthetic embedding traffic for the codec's tests and benchmark.

This module only *makes inputs*; it holds none of the codec's arithmetic.  The
same tensors feed the CUDA library and the CPU oracle.

The five workloads stand in for the Criteo Kaggle / Terabyte embedding traffic
that the method's evaluation uses ("Accelerating Communication in Deep Learning
Recommendation Model Training with Dual-Level Adaptive Lossy Compression",
§IV-A: 26 categorical features, fp32 embedding vectors, Zipf-skewed lookups);
the datasets themselves are not used.

All randomness is counter based: every value is a pure function of
(seed, stream, table, row, dim), so only the gathered rows are materialised and
the CPU and CUDA builds of a tensor are bit-identical (integer mixing, then
exactly-rounded float32 operations in a fixed order).

Workloads (B = batch, T = tables, D = embedding dim):
  tiny   [512, 4, 16]     1,000 rows/table, U(+-1/sqrt(1000)), Zipf s=1.05, eb = 1e-3 abs
  fwd    [8192, 26, 128]  rows_t = floor(10^(3+3u_t)), U(+-1/sqrt(rows_t)), Zipf 1.05,
                          eb_t = 1e-2 * range of table t's gathered slice
  bwd    [8192, 26, 128]  gradients count(idx) * z[t, idx, :], z ~ N(0, 1e-4) per table row,
                          Zipf 1.2, eb_t = 1e-3 * 30^(t/25) abs (1e-3 .. 3e-2, log-spaced)
  sweep  fwd regenerated per iteration i (index seed = i), rows drifting by N(0, 1e-3) per
         step (marginal at step i: sqrt(i) * 1e-3 * z), base bound 3e-3 * range, decayed by
         the linear schedule m0 = 10 over 99 iterations (3e-2 -> 3e-3 of range)
  large  [65536, 26, 256] 10^6 rows/table, U(+-1e-3), Zipf 1.1, eb_t = 1e-2 * range;
         variant "bf16": the same values rounded to bfloat16 (RNE) and stored as fp32
N(0, sigma) is drawn as sigma * sqrt(3) * (u1 + u2 + u3 + u4 - 2) (Irwin-Hall, k = 4), which
uses only exactly-rounded operations.
"""
from __future__ import annotations

import dataclasses
import functools
import math

import numpy as np
import torch

M32 = 0xFFFFFFFF

# stream identifiers of the counter-based generator
_S_TABLE_ROWS, _S_INDEX, _S_VALUE, _S_NORMAL, _S_DRIFT = 1, 2, 3, 10, 20

SHAPES = {
    "tiny": (512, 4, 16),
    "fwd": (8192, 26, 128),
    "bwd": (8192, 26, 128),
    "sweep": (8192, 26, 128),
    "large": (65536, 26, 256),
}


def _mix(v):
    """32-bit integer mixer on Python ints or int64 tensors holding values < 2^32."""
    v = v ^ (v >> 16)
    v = (v * 0x21F0AAAD) & M32
    v = v ^ (v >> 15)
    v = (v * 0x735A2D97) & M32
    v = v ^ (v >> 15)
    return v


def _draw(seed: int, stream: int, *fields):
    """u32 counter-based draw keyed by (seed, stream, fields...)."""
    h = _mix((seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x165667B1) & M32)
    for f in fields:
        h = _mix((h ^ f) & M32) if isinstance(h, int) and isinstance(f, int) else _mix(h ^ f)
    return h


def _u01_f32(h: torch.Tensor) -> torch.Tensor:
    """Uniform float32 in [0, 1) with 24 bits, exact."""
    return (h >> 8).to(torch.float32) * (1.0 / 16777216.0)


@functools.lru_cache(maxsize=64)
def _zipf_cdf(n: int, s: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    c = np.cumsum(k ** (-s))
    return c / c[-1]


def zipf_indices(n: int, s: float, seed: int, t: int, B: int) -> np.ndarray:
    """B row indices in [0, n) with P(row r) proportional to (r+1)^-s."""
    b = torch.arange(B, dtype=torch.int64)
    u = _draw(seed, _S_INDEX, t, b).numpy().astype(np.float64) * (1.0 / 4294967296.0)
    idx = np.searchsorted(_zipf_cdf(n, s), u, side="right")
    return np.minimum(idx, n - 1).astype(np.int64)


def table_rows(seed: int, T: int):
    """rows_t = floor(10^(3 + 3 u_t)): log-uniform over 10^3 .. 10^6."""
    out = []
    for t in range(T):
        u = _draw(seed, _S_TABLE_ROWS, t) / 4294967296.0
        out.append(int(math.floor(10.0 ** (3.0 + 3.0 * u))))
    return out


def _uniform_rows(seed, t, idx, D, amp, device):
    d = torch.arange(D, dtype=torch.int64, device=device)[None, :]
    r = idx[:, None]
    u = _u01_f32(_draw(seed, _S_VALUE, t, r, d))
    return (u * 2.0 - 1.0) * torch.tensor(amp, dtype=torch.float32, device=device)


def _normal_rows(seed, stream, t, idx, D, sigma, device):
    d = torch.arange(D, dtype=torch.int64, device=device)[None, :]
    r = idx[:, None]
    acc = _u01_f32(_draw(seed, stream, t, r, d))
    for j in range(1, 4):
        acc = acc + _u01_f32(_draw(seed, stream + j, t, r, d))
    scale = torch.tensor(sigma * math.sqrt(3.0), dtype=torch.float32, device=device)
    return (acc - 2.0) * scale


def _range_bound(x: torch.Tensor, rel: float) -> torch.Tensor:
    """eb_t = rel * (max - min) over table t's gathered [B, D] slice, float32."""
    B, T, D = x.shape
    xt = x.permute(1, 0, 2).reshape(T, -1)
    rng = (xt.max(dim=1).values - xt.min(dim=1).values).to(torch.float32)
    out = (rng * torch.tensor(rel, dtype=torch.float32, device=x.device)).cpu()
    # a constant table would give eb = 0; give it the smallest usable bound
    return torch.where(out > 0, out, torch.full_like(out, 1e-30))


@dataclasses.dataclass
class Workload:
    name: str
    x: torch.Tensor            # [B, T, D] float32, contiguous
    eb: torch.Tensor           # [T] float32 absolute bounds (CPU); for "sweep", the base bounds
    indices: np.ndarray        # [B, T] gathered row ids
    schedule: dict | None = None  # for "sweep": base bounds and decay parameters

    @property
    def shape(self):
        return tuple(self.x.shape)

    @property
    def nbytes(self) -> int:
        return self.x.numel() * 4


def make(name: str, *, device="cpu", iteration: int = 0, batch: int | None = None,
         tables: int | None = None, variant: str | None = None, seed: int = 0) -> Workload:
    """Build one workload; batch / tables shrink it with the same distributions."""
    if name not in SHAPES:
        raise KeyError(name)
    B, T, D = SHAPES[name]
    B = batch if batch is not None else B
    T = tables if tables is not None else T
    dev = torch.device(device)
    x = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    idx_all = np.zeros((B, T), dtype=np.int64)
    schedule = None
    if name == "tiny":
        for t in range(T):
            idx = zipf_indices(1000, 1.05, seed, t, B)
            idx_all[:, t] = idx
            x[:, t, :] = _uniform_rows(seed, t, torch.from_numpy(idx).to(dev), D, 1.0 / math.sqrt(1000.0), dev)
        eb = torch.full((T,), 1e-3, dtype=torch.float32)
    elif name in ("fwd", "sweep"):
        rows = table_rows(seed, T)
        iseed = seed + iteration if name == "sweep" else seed
        for t in range(T):
            idx = zipf_indices(rows[t], 1.05, iseed, t, B)
            idx_all[:, t] = idx
            it = torch.from_numpy(idx).to(dev)
            v = _uniform_rows(seed, t, it, D, 1.0 / math.sqrt(rows[t]), dev)
            if name == "sweep" and iteration > 0:
                v = v + _normal_rows(seed + iteration, _S_DRIFT, t, it, D, 1e-3 * math.sqrt(iteration), dev)
            x[:, t, :] = v
        if name == "fwd":
            eb = _range_bound(x, 1e-2)
        else:
            base = _range_bound(x, 3e-3)
            # the caller applies the decay schedule to these base bounds
            schedule = {"base": base, "fn": "linear", "m0": 10.0, "phase_len": 99, "n_steps": 1,
                        "iteration": iteration}
            eb = base
    elif name == "bwd":
        rows = table_rows(seed, T)
        for t in range(T):
            idx = zipf_indices(rows[t], 1.2, seed, t, B)
            idx_all[:, t] = idx
            it = torch.from_numpy(idx).to(dev)
            _, inv, cnt = torch.unique(it, return_inverse=True, return_counts=True)
            count = cnt[inv].to(torch.float32)[:, None]
            # variant "s1e-2": sigma 1e-2, the robustness case with heavy tails past the 8-bit bins
            sigma = 1e-2 if variant == "s1e-2" else 1e-4
            x[:, t, :] = _normal_rows(seed, _S_NORMAL, t, it, D, sigma, dev) * count
        eb = torch.tensor([1e-3 * 30.0 ** (t / 25.0) for t in range(T)], dtype=torch.float32)
    elif name == "large":
        for t in range(T):
            idx = zipf_indices(1000000, 1.1, seed, t, B)
            idx_all[:, t] = idx
            v = _uniform_rows(seed, t, torch.from_numpy(idx).to(dev), D, 1e-3, dev)
            if variant == "bf16":
                v = v.to(torch.bfloat16).to(torch.float32)
            x[:, t, :] = v
        eb = _range_bound(x, 1e-2)
    return Workload(name=name if variant is None else f"{name}-{variant}", x=x.contiguous(), eb=eb,
                    indices=idx_all, schedule=schedule)

