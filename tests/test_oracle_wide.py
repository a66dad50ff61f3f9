"""Pins of the oracle's wide alphabet (radius 512: bins q in (-512, 512),
1024 symbols, 16-bit codes).  The paper ("Accelerating Communication in Deep
Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-D quantization encoder and Huffman encoder) fixes no radius;
this option widens the bins so that heavy-tailed values stop being outliers.
Pinned against hand-computed codes, the 8-bit alphabet where both apply, a
textbook heap Huffman and the Kraft equality over 1024 symbols, brute-force
dedup, the error bound, and the container layout."""
import heapq
from fractions import Fraction

import numpy as np
import pytest

import oracle as o
import workloads


def _u32(buf, off):
    return int.from_bytes(bytes(buf[off:off + 4]), "little")


def _u64(buf, off):
    return int.from_bytes(bytes(buf[off:off + 8]), "little")


def test_quantize_hand_values():
    # eb = 0.5: bins of width 1 on the integers, q = round_half_even(x), symbol q + 512
    x = np.array([0.0, -0.0, 1.0, -1.0, 128.0, -128.0, 200.0, 511.0, -511.0, 511.5, -511.5, 512.0,
                  510.5, 2.5, -2.5, np.nan, np.inf, -np.inf, 1e30, 127.5], np.float32)
    want = [512, 512, 513, 511, 640, 384, 712, 1023, 1, 0, 0, 0,
            1022, 514, 510, 0, 0, 0, 0, 640]
    assert o.quantize_r(x, 0.5, 512).tolist() == want
    # the same inputs with radius 128: everything at or past 128 bins is an outlier
    assert o.quantize_r(x, 0.5, 128).tolist() == o.quantize(x, 0.5).tolist()


def test_wide_agrees_with_narrow_inside_the_narrow_range():
    rng = np.random.default_rng(4)
    eb = float(np.float32(1e-3))
    x = (rng.standard_normal(50000) * 300 * eb).astype(np.float32)
    n = o.quantize(x, eb).astype(np.int64)
    w = o.quantize_r(x, eb, 512).astype(np.int64)
    both = (n != 0) & (w != 0)
    assert (n[both] - 128 == w[both] - 512).all()
    # every wide outlier is a narrow one, and the wide alphabet has far fewer
    assert ((w == 0) <= (n == 0)).all()
    assert (w == 0).sum() * 4 < (n == 0).sum()
    # reconstruction keeps the bound: |x - (sym - 512) * 2 eb| <= eb
    lit = w != 0
    xh = ((w[lit] - 512).astype(np.float32) * np.float32(2 * eb)).astype(np.float32)
    assert (np.abs(x[lit].astype(np.float64) - xh.astype(np.float64)) <= eb).all()


def _heap_cost(freq):
    f = [int(v) for v in freq if v > 0]
    if len(f) <= 1:
        return sum(f)
    heapq.heapify(f)
    cost = 0
    while len(f) > 1:
        a, b = heapq.heappop(f), heapq.heappop(f)
        cost += a + b
        heapq.heappush(f, a + b)
    return cost


@pytest.mark.parametrize("n,kind", [(2, "u"), (300, "u"), (700, "g"), (1024, "u"), (1024, "g"), (1000, "s")])
def test_huffman_over_1024_symbols(n, kind):
    rng = np.random.default_rng(n)
    f = np.zeros(1024, np.uint64)
    syms = rng.choice(1024, n, replace=False)
    if kind == "u":
        f[syms] = rng.integers(1, 1000, n)
    elif kind == "g":
        f[syms] = (2.0 ** rng.uniform(0, 14, n)).astype(np.int64) + 1
    else:
        f[syms] = rng.integers(1, 3, n)
    lens, rounds = o.huffman_lengths(f, symbols=1024)
    assert rounds == 0
    assert ((lens > 0) == (f > 0)).all()
    if n >= 2:
        assert sum(Fraction(1, 2 ** int(v)) for v in lens if v) == 1
    assert int((f * lens.astype(np.uint64)).sum()) == _heap_cost(f)
    codes = o.canonical_codes(lens)
    words = sorted(format(int(c), f"0{int(l)}b") for c, l in zip(codes, lens) if l)
    assert all(not b.startswith(a) for a, b in zip(words, words[1:]))   # prefix-free


def test_huffman_length_limit_over_1024_symbols():
    fib = [1, 1]
    while len(fib) < 40:
        fib.append(fib[-1] + fib[-2])
    f = np.zeros(1024, np.uint64)
    f[600:640] = fib                     # a depth-39 tree: the limit must act
    lens, rounds = o.huffman_lengths(f, symbols=1024)
    assert rounds >= 1 and lens.max() <= 24
    assert sum(Fraction(1, 2 ** int(v)) for v in lens if v) == 1
    lens32, r32 = o.huffman_lengths(f, lmax=32, symbols=1024)
    assert lens32.max() > 24


def test_key_of_the_narrow_alphabet_is_unchanged():
    rng = np.random.default_rng(2)
    for D in (4, 16, 128):
        s = rng.integers(0, 256, D).astype(np.uint8)
        x = rng.standard_normal(D).astype(np.float32)
        assert o.vector_hash(s, x) == int(o._lib().ebo_vector_hash_r(o._ptr(s.astype(np.uint16)), o._ptr(x), D, 128))


def _rows(pattern, D=8, big=300.0):
    # rows keyed by a letter, values around `big` bins (outliers in the 8-bit alphabet)
    base = {c: (np.arange(D, dtype=np.float32) + big + 3 * k) for k, c in enumerate(sorted(set(pattern)))}
    return np.stack([base[c] for c in pattern])[:, None, :].astype(np.float32), np.array([0.5], np.float32)


def test_container_layout_and_round_trip():
    x, eb = _rows("ABAACB")
    buf, info, sym, ref, lens = o.compress(x, eb, want_internals=True, radius=512)
    assert _u32(buf, 24) == 512
    assert _u64(buf, 88) == 144 + 1 * (16 + 1024)               # one table record of 1040 bytes
    assert sym.dtype == np.uint16 and lens.shape == (1, 1024)
    assert info["n_outlier"] == 0 and info["n_match"] == 3
    assert ref[0].tolist() == [0, 1, 0, 0, 4, 1]
    xh, s2 = o.decompress(buf, *x.shape)
    assert np.array_equal(xh, x)                                 # integers on the bin centres
    assert np.array_equal(s2, sym)
    # the 8-bit alphabet codes all of these values as outliers
    _, info8 = o.compress(x, eb)
    assert info8["n_outlier"] == x.size - 3 * 8


def test_dedup_brute_force():
    rng = np.random.default_rng(8)
    pool = (rng.integers(-600, 600, size=(5, 3, 8)) * 1.0).astype(np.float32)
    x = np.ascontiguousarray(pool[rng.integers(0, 5, size=60)])
    x[7, 1, 3] = np.nan                                          # an outlier row too
    eb = np.full(3, 0.5, np.float32)
    _, info, sym, ref, _ = o.compress(x, eb, want_internals=True, radius=512)
    want = 0
    for t in range(3):
        for b in range(60):
            earlier = [r for r in range(b) if np.array_equal(x[r, t].view(np.uint32), x[b, t].view(np.uint32))]
            if earlier:
                want += 1
                assert ref[t, b] == earlier[0]
    assert info["n_match"] == want


def test_error_bound_modes_window_and_chunks():
    wl = workloads.make("bwd", batch=700, tables=5, variant="s1e-2")
    x, eb = wl.x.numpy(), wl.eb.numpy()
    base, _ = o.compress(x, eb, radius=512)
    xb = o.decompress(base, *x.shape)[0]
    err = np.abs(x.astype(np.float64) - xb.astype(np.float64))
    assert (err <= eb.astype(np.float64)[None, :, None]).all()
    # raw codes are 10 bits; every mode and window restores the same values
    buf, _, _, _, lens = o.compress(x, eb, want_internals=True, radius=512, modes=np.array([3] * 5, np.uint8))
    assert (lens == 10).all()
    for kw in ({"modes": np.array([0, 1, 2, 3, 1], np.uint8)}, {"window": 16}):
        b2, _ = o.compress(x, eb, radius=512, **kw)
        assert np.array_equal(o.decompress(b2, *x.shape)[0].view(np.uint32), xb.view(np.uint32))
    cb, offs = o.compress_chunked(x, eb, 3, radius=512)
    assert np.array_equal(o.decompress_chunked(cb, offs, *x.shape).view(np.uint32), xb.view(np.uint32))


def test_bad_radius_field():
    x, eb = _rows("AB")
    buf, _ = o.compress(x, eb, radius=512)
    for r in (0, 256, 1024):
        b = buf.copy()
        b[24:28] = np.frombuffer(np.uint32(r).tobytes(), np.uint8)
        rc, _, _ = o.decompress_rc(b, *x.shape)
        assert rc == o.ERR_CORRUPT
    with pytest.raises(ValueError):
        o.quantize_r(x, 0.5, 256)
