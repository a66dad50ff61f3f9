"""Pins of the oracle's per-table hybrid modes, the Homogenization Index
(Eq. 1) and the Eq. (2) compressor selection.

Method: "Accelerating Communication in Deep Learning Recommendation Model
Training with Dual-Level Adaptive Lossy Compression" (arXiv 2407.04272),
§III-C Eq. (1), §III-D "Selection Between Two Encoders" and Eq. (2),
Tables III and IV.
"""
import os

import numpy as np
import pytest

import oracle as o
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "homo_index_tables.txt")


def _rows():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        tab, eb, n_ori, n_q, batch, printed = line.split()
        rows.append((int(n_ori), int(n_q), int(batch), float(printed)))
    return rows


def test_homo_index_matches_tables_iii_and_iv():
    rows = _rows()
    assert len(rows) == 16
    for n_ori, n_q, batch, printed in rows:
        eta = o.homo_index(n_ori, n_q)
        assert 0.0 <= eta <= 1.0
        # the tables print N_quantized / N_original = 1 - eta, rounded to 6 decimals
        assert abs((1.0 - eta) - printed) <= 5e-7, (n_ori, n_q, printed, eta)
        assert n_q <= n_ori <= batch


def test_homo_index_definition_endpoints():
    assert o.homo_index(1000, 1000) == 0.0          # no homogenization
    assert o.homo_index(1000, 1) == pytest.approx(0.999)   # all but one merged
    assert o.homo_index(0, 0) == 0.0
    assert o.homo_index(110, 68) == pytest.approx(42 / 110, rel=1e-15)


def test_speedup_closed_forms():
    # 1 / (1/4 + 10 (1/100 + 1/200)) = 1 / (0.25 + 0.15) = 2.5
    assert o.speedup(4.0, 10.0, 100.0, 200.0) == pytest.approx(2.5, rel=1e-15)
    # infinitely fast codecs: the compression ratio itself
    assert o.speedup(7.0, 0.0, 1.0, 1.0) == pytest.approx(7.0, rel=1e-15)
    # CR 1 and free codecs: no gain
    assert o.speedup(1.0, 0.0, 5.0, 5.0) == pytest.approx(1.0)
    # slow codecs lose against no compression even at a high ratio
    assert o.speedup(100.0, 100.0, 10.0, 10.0) < 1.0
    assert o.speedup(0.0, 1.0, 1.0, 1.0) == 0.0
    assert o.speedup(2.0, 1.0, 0.0, 1.0) == 0.0


def test_speedup_monotone():
    rng = np.random.default_rng(3)
    for _ in range(200):
        cr, bw, tc, td = rng.uniform(0.5, 50), rng.uniform(0, 100), rng.uniform(1, 1000), rng.uniform(1, 1000)
        s = o.speedup(cr, bw, tc, td)
        assert o.speedup(cr * 1.5, bw, tc, td) > s
        assert o.speedup(cr, bw * 1.5 + 1, tc, td) < s
        assert o.speedup(cr, bw, tc * 2, td) > s or bw == 0


def test_select_modes_hand_example():
    # two candidates: A (CR 10, slow) and B (CR 5, fast); link 1 unit/s
    tc = [2.0, 50.0]
    td = [2.0, 50.0]
    cr = [[10.0, 5.0],      # A: 1/(0.1 + 1) = 0.909;  B: 1/(0.2 + 0.04) = 4.17  -> B
          [1000.0, 1.0]]    # A: 1/(0.001 + 1) = 0.999; B: 1/(1 + 0.04) = 0.962 -> A
    assert o.select_modes(cr, tc, td, 1.0).tolist() == [1, 0]
    # on a free link the higher ratio always wins
    assert o.select_modes(cr, tc, td, 0.0).tolist() == [0, 0]
    # ties go to the lower index
    assert o.select_modes([[3.0, 3.0]], [1.0, 1.0], [1.0, 1.0], 0.5).tolist() == [0]


def _modes(T, m):
    return np.full(T, m, np.uint8)


@pytest.mark.parametrize("name", ["tiny", "bwd"])
def test_modes_keep_reconstruction_and_bound(name):
    wl = workloads.make(name, batch=512)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    T = x.shape[1]
    ref = None
    for m in range(4):
        buf, info, sym, refv, lens = o.compress(x, eb, want_internals=True, modes=_modes(T, m))
        xh, _ = o.decompress(buf, *x.shape)
        if ref is None:
            ref = xh
        # the same quantization in every mode: dedup and entropy coding are lossless
        assert np.array_equal(xh.view(np.uint32), ref.view(np.uint32))
        if m & 1:   # no dedup: every vector a literal
            assert info["n_match"] == 0
            assert (refv == np.arange(x.shape[0], dtype=np.uint32)[None, :]).all()
        if m & 2:   # raw codes: all lengths 8
            assert (lens == 8).all()
            lit = refv == np.arange(x.shape[0], dtype=np.uint32)[None, :]
            n_code = int(lit.sum()) * x.shape[2]
            n_out = int(((sym == 0) & lit[:, :, None]).sum())
            bits = 8 * n_code + 32 * n_out
            # per-segment bitstreams are padded to 128 bits; the payload is the closed form
            assert info["bitstream_bytes"] * 8 >= bits
            assert info["bitstream_bytes"] * 8 - bits < 128 * T * ((x.shape[0] + 511) // 32 + 1)


def test_raw_codes_are_the_symbols():
    # raw mode: an outlier-free literal row is stored as its code bytes, MSB-first
    rng = np.random.default_rng(5)
    B, T, D = 64, 1, 16
    x = rng.uniform(-0.1, 0.1, size=(B, T, D)).astype(np.float32)
    eb = np.array([1e-2], np.float32)
    buf, info, sym, refv, lens = o.compress(x, eb, want_internals=True, modes=[3])
    assert info["n_outlier"] == 0 and info["n_match"] == 0
    off_bits = int.from_bytes(bytes(buf[120:128]), "little")
    words = np.frombuffer(bytes(buf[off_bits:]), dtype="<u4")
    stream = b"".join(int(wd).to_bytes(4, "big") for wd in words)
    assert stream[: B * D] == sym[0].reshape(-1).tobytes()


def test_invalid_mode_rejected():
    wl = workloads.make("tiny")
    with pytest.raises(RuntimeError):
        o.compress(wl.x.numpy(), wl.eb.numpy(), modes=np.full(wl.x.shape[1], 4, np.uint8))


def test_mode_zero_is_the_default():
    wl = workloads.make("tiny")
    a, _ = o.compress(wl.x.numpy(), wl.eb.numpy())
    b, _ = o.compress(wl.x.numpy(), wl.eb.numpy(), modes=np.zeros(wl.x.shape[1], np.uint8))
    assert np.array_equal(a, b)
