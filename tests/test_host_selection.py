"""The C ABI's host-side Eq. (1) / Eq. (2) functions against the oracle's and
against the values Tables III and IV print ("Accelerating Communication in
Deep Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-C Eq. (1), §III-D Eq. (2)).  No GPU needed."""
import ctypes
import os

import numpy as np
import pytest

import error_bounded_lossy_gb300 as ebc
import oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "homo_index_tables.txt")


def _lib_or_skip():
    try:
        return ebc.lib()
    except RuntimeError as e:   # library not built here
        pytest.skip(str(e))


def test_homo_index_tables():
    _lib_or_skip()
    n = 0
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        _, _, n_ori, n_q, _, printed = line.split()
        eta = ebc.ebc_homo_index(int(n_ori), int(n_q))
        assert eta == o.homo_index(int(n_ori), int(n_q))
        assert abs((1.0 - eta) - float(printed)) <= 5e-7
        n += 1
    assert n == 16


def test_speedup_matches_oracle():
    _lib_or_skip()
    rng = np.random.default_rng(11)
    for _ in range(500):
        args = (rng.uniform(0.1, 100), rng.uniform(0, 50), rng.uniform(0.1, 1000), rng.uniform(0.1, 1000))
        assert ebc.ebc_speedup(*args) == pytest.approx(o.speedup(*args), rel=1e-15)
    assert ebc.ebc_speedup(4.0, 10.0, 100.0, 200.0) == pytest.approx(2.5, rel=1e-15)
    assert ebc.ebc_speedup(0.0, 1.0, 1.0, 1.0) == 0.0


def test_select_modes_matches_oracle():
    _lib_or_skip()
    rng = np.random.default_rng(12)
    for T, M in [(1, 1), (5, 2), (26, 4), (100, 3)]:
        cr = rng.uniform(0.5, 40, size=(T, M))
        tc = rng.uniform(10, 500, size=M)
        td = rng.uniform(10, 500, size=M)
        bw = float(rng.uniform(0, 30))
        out = np.zeros(T, np.uint8)
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        assert ebc.ebc_select_modes(p(cr), p(tc), p(td), bw, T, M, p(out)) == ebc.EBC_OK
        assert out.tolist() == o.select_modes(cr, tc, td, bw).tolist()
    assert ebc.ebc_select_modes(None, None, None, 1.0, 3, 2, None) == ebc.EBC_ERR_INVALID_ARG
