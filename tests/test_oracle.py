"""Pins of the CPU oracle against what the method and the mathematics fix.

Each test checks the oracle against something other than itself: the error
bound of the quantization encoder, nearest-bin optimality, a textbook heap
Huffman and brute-force optimal prefix codes, the Kraft equality, prefix
freedom, brute-force first-occurrence dedup, closed forms of the decay
schedule, a container worked out by hand, and the round trip.

Method: "Accelerating Communication in Deep Learning Recommendation Model
Training with Dual-Level Adaptive Lossy Compression" (§III-C schedule, §III-D
quantization + vector-based LZ + Huffman, §III-E single-buffer layout).
"""
import heapq
import itertools
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle as o
import workloads


# ---------------------------------------------------------------- quantization
def test_quantize_special_values():
    # eb = 0.5 -> bins of width 1 centred on the integers (q = round_half_even(x))
    x = np.array([0.0, -0.0, 1.0, -1.0, 2.5, 3.5, -2.5, 127.0, -127.0, 127.5, -127.5, 128.0,
                  1e30, np.inf, -np.inf, np.nan, 0.5, -0.5, 1.5, 126.49], np.float32)
    want = [128, 128, 129, 127, 130, 132, 126, 255, 1, 0, 0, 0,
            0, 0, 0, 0, 128, 128, 130, 254]
    assert o.quantize(x, 0.5).tolist() == want


def _exact_err(x, xhat):
    return abs(Fraction(float(x)) - Fraction(float(xhat)))


@pytest.mark.parametrize("eb", [1e-3, 3.7e-2, 0.25, 1e-6])
def test_quantize_bound_and_nearest_bin(eb):
    rng = np.random.default_rng(7)
    eb = float(np.float32(eb))
    x = (rng.standard_normal(20000) * 40 * eb).astype(np.float32)
    x[:50] = (np.arange(50) - 25).astype(np.float32) * np.float32(2 * eb)  # bin centres
    x[50:100] = ((np.arange(50) - 25) + 0.5).astype(np.float32) * np.float32(2 * eb)  # half bins
    sym = o.quantize(x, eb)
    lit = sym != 0
    xhat = np.array([o.dequantize(int(s), eb) for s in sym[lit]], np.float32)
    # |x - xhat| <= eb, exactly (float64 subtraction of two nearby float32 is exact)
    err = np.abs(x[lit].astype(np.float64) - xhat.astype(np.float64))
    assert (err <= eb).all()
    # the exact check on a sample, in rationals
    for xi, xh in list(zip(x[lit], xhat))[:300]:
        assert _exact_err(xi, xh) <= Fraction(eb)
    # nearest bin: no neighbouring bin centre is closer by more than rounding noise
    q = sym[lit].astype(np.int64) - 128
    c = Fraction(float(np.float32(2 * eb)))
    for xi, qi in list(zip(x[lit], q))[:2000]:
        d0 = abs(Fraction(float(xi)) - qi * c)
        for nb in (qi - 1, qi + 1):
            assert d0 <= abs(Fraction(float(xi)) - nb * c) + c * Fraction(1, 1 << 20)
    # every value inside the code range is coded, except exact half-bin points, where the
    # even bin is tried and its fp32 reconstruction can sit just beyond eb (kept raw then)
    t = x.astype(np.float64) / float(np.float32(2 * eb))
    inside = np.abs(t) < 120
    half = np.abs(np.abs(t) % 1.0 - 0.5) < 1e-4
    assert (sym[inside & ~half] != 0).all()
    assert (sym[np.abs(t) > 127.6] == 0).all()


def test_quantize_outlier_range_exact():
    eb = 0.5
    x = np.array([126.5, 126.51, 127.49, 127.5, -127.49, -127.5, -127.51], np.float32)
    # |q| must stay below R = 128
    assert o.quantize(x, eb).tolist() == [254, 255, 255, 0, 1, 0, 0]


def test_quantize_rejects_bad_bounds():
    for eb in [0.0, -1.0, float("nan"), float("inf"), 1e-45, 3e38]:
        with pytest.raises(ValueError):
            o.quantize(np.zeros(4, np.float32), eb)


# ---------------------------------------------------------------- Huffman
def heap_huffman_cost(freq):
    """Textbook Huffman with a binary heap: returns the optimal total bits."""
    f = [int(v) for v in freq if v > 0]
    if len(f) <= 1:
        return sum(f)
    h = list(f)
    heapq.heapify(h)
    cost = 0
    while len(h) > 1:
        a = heapq.heappop(h)
        b = heapq.heappop(h)
        cost += a + b
        heapq.heappush(h, a + b)
    return cost


def brute_force_optimal_cost(freq, max_len=6):
    f = [int(v) for v in freq if v > 0]
    best = None
    for lens in itertools.product(range(1, max_len + 1), repeat=len(f)):
        if sum(Fraction(1, 2 ** l) for l in lens) <= 1:
            c = sum(a * l for a, l in zip(f, lens))
            best = c if best is None else min(best, c)
    return best


def kraft_sum(lens):
    return sum(Fraction(1, 2 ** int(l)) for l in lens if l > 0)


def _random_hists():
    rng = np.random.default_rng(11)
    out = []
    for n in [2, 3, 5, 17, 64, 200, 256]:
        for kind in ("uniform", "geometric", "gauss", "sparse"):
            f = np.zeros(256, np.uint64)
            syms = rng.choice(256, n, replace=False)
            if kind == "uniform":
                v = rng.integers(1, 1000, n)
            elif kind == "geometric":
                v = (2.0 ** rng.uniform(0, 20, n)).astype(np.int64) + 1
            elif kind == "gauss":
                v = (1e6 * np.exp(-0.5 * ((np.arange(n) - n / 2) / (n / 8 + 1)) ** 2)).astype(np.int64) + 1
            else:
                v = rng.integers(1, 3, n)
            f[syms] = v
            out.append(f)
    return out


@pytest.mark.parametrize("f", _random_hists())
def test_huffman_optimal_and_complete(f):
    lens, rounds = o.huffman_lengths(f)
    assert rounds == 0
    assert ((lens > 0) == (f > 0)).all()
    assert kraft_sum(lens) == 1                      # complete prefix code
    assert int((f * lens.astype(np.uint64)).sum()) == heap_huffman_cost(f)


@pytest.mark.parametrize("seed", range(12))
def test_huffman_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 6))
    f = np.zeros(256, np.uint64)
    f[rng.choice(256, n, replace=False)] = rng.integers(1, 50, n)
    lens, _ = o.huffman_lengths(f)
    assert int((f * lens.astype(np.uint64)).sum()) == brute_force_optimal_cost(f[f > 0])


def test_huffman_degenerate():
    f = np.zeros(256, np.uint64)
    lens, _ = o.huffman_lengths(f)
    assert (lens == 0).all()
    f[77] = 5
    lens, _ = o.huffman_lengths(f)
    assert lens[77] == 1 and lens.sum() == 1
    f[3] = 1
    lens, _ = o.huffman_lengths(f)
    assert lens[77] == 1 and lens[3] == 1


def test_huffman_length_limit():
    # Fibonacci weights give a depth-(n-1) Huffman tree: 30 symbols -> 29 > 24
    fib = [1, 1]
    while len(fib) < 30:
        fib.append(fib[-1] + fib[-2])
    f = np.zeros(256, np.uint64)
    f[:30] = fib
    lens, rounds = o.huffman_lengths(f)
    assert rounds >= 1
    assert lens.max() <= 24
    assert kraft_sum(lens) == 1
    lens_unlimited, r2 = o.huffman_lengths(f, lmax=32)
    assert r2 == 0 and lens_unlimited.max() == 29


@pytest.mark.parametrize("f", _random_hists()[::3])
def test_canonical_codes_prefix_free_and_ordered(f):
    lens, _ = o.huffman_lengths(f)
    code = o.canonical_codes(lens)
    used = [s for s in range(256) if lens[s] > 0]
    words = {s: format(int(code[s]), "0%db" % int(lens[s])) for s in used}
    for a in used:
        for b in used:
            if a != b:
                assert not words[b].startswith(words[a])
    # canonical order: (length, symbol) ascending <=> left-aligned code ascending
    order = sorted(used, key=lambda s: (lens[s], s))
    vals = [int(code[s]) << (24 - int(lens[s])) for s in order]
    assert vals == sorted(vals) and len(set(vals)) == len(vals)
    assert vals[0] == 0


def test_canonical_rejects_over_full():
    lens = np.zeros(256, np.uint8)
    lens[:3] = 1
    with pytest.raises(ValueError):
        o.canonical_codes(lens)


# ---------------------------------------------------------------- schedule
@pytest.mark.parametrize("fn", ["linear", "stepwise", "drop", "log"])
def test_decay_endpoints_and_monotone(fn):
    m0, P = 3.0, 40
    assert o.decay_factor(fn, 0, m0, P, 4) == m0
    assert o.decay_factor(fn, P, m0, P, 4) == 1.0
    assert o.decay_factor(fn, 10 * P, m0, P, 4) == 1.0
    vals = [o.decay_factor(fn, i, m0, P, 4) for i in range(P + 5)]
    assert all(a >= b for a, b in zip(vals, vals[1:]))
    assert o.decay_factor("none", 3, m0, P, 4) == 1.0


def test_decay_closed_forms():
    # logarithmic: geometric interpolation, sqrt(m0) half-way
    assert o.decay_factor("log", 50, 4.0, 100) == pytest.approx(2.0, rel=1e-15)
    # stepwise: S + 1 distinct values m0 - (m0 - 1) k / S
    vals = {o.decay_factor("stepwise", i, 5.0, 100, 4) for i in range(0, 101)}
    assert vals == {5.0, 4.0, 3.0, 2.0, 1.0}
    # linear midpoint
    assert o.decay_factor("linear", 50, 3.0, 100) == 2.0
    # "Decay_2x" and "Drop_2x" of the iteration-wise experiment: 2x base down to base
    assert o.decay_factor("linear", 0, 2.0, 10) == 2.0 and o.decay_factor("linear", 10, 2.0, 10) == 1.0
    assert [o.decay_factor("drop", i, 2.0, 10) for i in (0, 9, 10, 11)] == [2.0, 2.0, 1.0, 1.0]
    # the sweep workload: 3e-2 -> 3e-3 of range with base 3e-3 of range
    base = np.array([3e-3], np.float32)
    assert o.scheduled_bounds(base, "linear", 0, 10.0, 99)[0] == np.float32(float(base[0]) * 10.0)
    assert o.scheduled_bounds(base, "linear", 99, 10.0, 99)[0] == np.float32(3e-3)


# ---------------------------------------------------------------- dedup
def brute_force_refs(sym, x):
    """First occurrence among vectors with identical codes and outlier bits."""
    T, B, D = sym.shape
    ref = np.zeros((T, B), np.uint32)
    xb = x.view(np.uint32)
    for t in range(T):
        for b in range(B):
            ref[t, b] = b
            for r in range(b):
                if (sym[t, r] == sym[t, b]).all():
                    out = sym[t, b] == 0
                    if (xb[r, t][out] == xb[b, t][out]).all():
                        ref[t, b] = r
                        break
    return ref


def _planted(B=96, T=3, D=16, seed=3):
    rng = np.random.default_rng(seed)
    eb = np.array([1e-2, 2e-2, 5e-3], np.float32)[:T]
    x = (rng.uniform(-1, 1, (B, T, D)) * 0.3).astype(np.float32)
    for t in range(T):
        for b in range(B):
            if rng.uniform() < 0.5 and b > 0:
                src = int(rng.integers(0, b))
                if rng.uniform() < 0.5:
                    x[b, t] = x[src, t]                         # exact repeat
                else:                                           # homogenized repeat
                    c = np.round(x[src, t] / (2 * eb[t])) * (2 * eb[t])
                    x[src, t] = c.astype(np.float32)
                    x[b, t] = (c + rng.uniform(-0.2, 0.2, D) * eb[t]).astype(np.float32)
    x[5, 0, 3] = np.float32(1e9)                               # outliers
    x[9, 0] = x[5, 0]
    x[11, 0] = x[5, 0]
    x[11, 0, 3] = np.float32(2e9)                              # same codes, other raw bits
    return x, eb


def test_dedup_matches_brute_force():
    x, eb = _planted()
    buf, info, sym, ref, lens = o.compress(x, eb, want_internals=True)
    assert (ref == brute_force_refs(sym, x)).all()
    assert ref[0, 9] == 5 and ref[0, 11] == 11
    # no hash collisions among distinct vectors in this input
    T, B, D = sym.shape
    for t in range(T):
        seen = {}
        for b in range(B):
            key = (sym[t, b].tobytes(), x[b, t][sym[t, b] == 0].tobytes())
            h = o.vector_hash(sym[t, b], x[b, t])
            assert seen.setdefault(h, key) == key
    assert info["n_match"] == int((ref != np.arange(B)[None, :]).sum())


def test_identical_rows_reconstruct_identically():
    x, eb = _planted(seed=5)
    buf, info = o.compress(x, eb)
    xh, _ = o.decompress(buf, *x.shape)
    B, T, D = x.shape
    for t in range(T):
        rows = {}
        for b in range(B):
            k = x[b, t].tobytes()
            if k in rows:
                assert xh[b, t].tobytes() == xh[rows[k], t].tobytes()
            rows.setdefault(k, b)


def test_hash_is_a_function_of_tokens():
    rng = np.random.default_rng(1)
    s = rng.integers(1, 256, 64).astype(np.uint8)
    xa = rng.standard_normal(64).astype(np.float32)
    xb = rng.standard_normal(64).astype(np.float32)
    assert o.vector_hash(s, xa) == o.vector_hash(s, xb)    # raw bits matter only at outliers
    s2 = s.copy()
    s2[10] ^= 1
    assert o.vector_hash(s2, xa) != o.vector_hash(s, xa)
    s[7] = 0
    xb[7] = xa[7] + 1
    assert o.vector_hash(s, xa) != o.vector_hash(s, xb)


# ---------------------------------------------------------------- container
def test_container_worked_by_hand():
    # B=2, T=1, D=4, eb=0.5 (bins = integers).  Row 0 codes: 0->128, 1->129, -1->127,
    # 0.5->128 (tie to even).  Row 1 repeats row 0: a match with ref 0.
    # Literal histogram {127:1, 128:2, 129:1}; leaves by (f, sym): 127, 129, 128.
    # Merge 127+129 -> node(2); then leaf 128 (2) ties node(2): leaf first -> root.
    # Lengths 128:1, 127:2, 129:2; canonical codes 128='0', 127='10', 129='11'.
    # Stream: 0 11 10 0 -> bits 011100 -> word 0x70000000, padded to 128 bits.
    # Layout: header 144, table record 272 -> segments at 416 (1 x 16 B), bitmap at 432
    # (1 word, padded to 16), chunk lengths at 448 (1 x u16 = 6), refs at 464 (u16 0),
    # bitstream at 480 (4 words), total 496.
    x = np.array([[[0.0, 1.0, -1.0, 0.5]], [[0.0, 1.0, -1.0, 0.5]]], np.float32)
    buf, info = o.compress(x, np.array([0.5], np.float32))
    assert len(buf) == 496
    hdr = struct.unpack_from("<4sIQIIIIIIIIQQQQQQQQQQQQ", buf.tobytes(), 0)
    assert hdr[0] == b"EBC1" and hdr[1] == 2 and hdr[2:5] == (2, 1, 4)
    assert hdr[5:11] == (128, 24, 2048, 32, 2, 0)
    assert hdr[11:16] == (1, 1, 0, 1, 4)                 # lit, match, outliers, chunks, words
    assert hdr[16:] == (416, 432, 448, 464, 480, 496, 0)
    b = buf.tobytes()
    assert struct.unpack_from("<fIII", b, 144) == (0.5, 1, 1, 0)
    lens = np.frombuffer(b, np.uint8, 256, 160)
    assert lens[127] == 2 and lens[128] == 1 and lens[129] == 2 and lens.sum() == 5
    assert struct.unpack_from("<IIII", b, 416) == (0, 0, 0, 6)   # word, chunk, match base; bits
    assert struct.unpack_from("<I", b, 432) == (0b10,)
    assert struct.unpack_from("<H", b, 448) == (6,)
    assert struct.unpack_from("<H", b, 464) == (0,)
    assert struct.unpack_from("<IIII", b, 480) == (0x70000000, 0, 0, 0)
    xh, sym = o.decompress(buf, 2, 1, 4)
    assert xh.tolist() == [[[0.0, 1.0, -1.0, 0.0]], [[0.0, 1.0, -1.0, 0.0]]]


def test_outlier_inline_worked_by_hand():
    # B=1, T=1, D=4, eb=0.5: codes 128, 0 (1000.0 is |q| >= 128), 129, 128.  Histogram
    # {0:1, 128:2, 129:1}; leaves by (f, sym): 0, 129, 128 -> 0+129 merge, then leaf 128 ties
    # the node and goes first: lengths 128:1, 0:2, 129:2; canonical 128='0', 0='10', 129='11'.
    # Stream: '0' + '10' + 32 raw bits of 1000.0 (0x447A0000) + '11' + '0' = 38 bits.
    x = np.array([[[0.0, 1000.0, 1.0, 0.0]]], np.float32)
    buf, info = o.compress(x, np.array([0.5], np.float32))
    # layout: header 144 + table 272 + segment 16 + bitmap 16 + chunks 16 + refs 0 -> bits at 464
    assert info["n_outlier"] == 1 and len(buf) == 480
    bits = "0" + "10" + format(0x447A0000, "032b") + "11" + "0"
    bits = bits.ljust(128, "0")
    words = [int(bits[i:i + 32], 2) for i in range(0, 128, 32)]
    assert struct.unpack_from("<IIII", buf.tobytes(), 464) == tuple(words)
    assert struct.unpack_from("<H", buf.tobytes(), 448) == (38,)
    xh, _ = o.decompress(buf, 1, 1, 4)
    assert xh.tolist() == [[[0.0, 1000.0, 1.0, 0.0]]]


@pytest.mark.parametrize("B,T,D", [(1, 1, 4), (33, 2, 8), (100, 3, 16), (70, 2, 32), (64, 1, 64),
                                   (65, 2, 128), (40, 2, 256), (33, 1, 512), (0, 3, 16), (5, 0, 16)])
def test_round_trip_shapes(B, T, D):
    rng = np.random.default_rng(B * 7 + D)
    x = (rng.standard_normal((B, T, D)) * 0.05).astype(np.float32)
    if B > 3:
        x[3] = x[1]
    if x.size:
        x.reshape(-1)[:: 97] = np.float32(50.0)     # a few outliers
    eb = np.full((T,), 1e-3, np.float32)
    buf, info, sym, ref, lens = o.compress(x, eb, want_internals=True)
    xh, sym2 = o.decompress(buf, B, T, D)
    assert (sym2 == sym).all()
    lit = sym != 0
    xt = x.transpose(1, 0, 2)
    xht = xh.transpose(1, 0, 2)
    assert (np.abs(xt[lit].astype(np.float64) - xht[lit]) <= 1e-3).all()
    assert (xt[~lit].view(np.uint32) == xht[~lit].view(np.uint32)).all()


def test_round_trip_nonfinite_bit_exact():
    x = np.zeros((8, 2, 16), np.float32)
    x[1, 0, :4] = [np.inf, -np.inf, np.nan, -np.nan]
    x.view(np.uint32)[2, 1, 5] = 0x7FC01234              # NaN payload
    x[3, 1, 7] = np.float32(1e-42)                       # subnormal
    buf, info = o.compress(x, np.array([1e-3, 1e-3], np.float32))
    xh, _ = o.decompress(buf, 8, 2, 16)
    assert xh.view(np.uint32)[1, 0, :4].tolist() == x.view(np.uint32)[1, 0, :4].tolist()
    assert xh.view(np.uint32)[2, 1, 5] == 0x7FC01234
    assert xh[3, 1, 7] == 0.0


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("fwd", {"batch": 300, "tables": 4}),
                                     ("bwd", {"batch": 300, "tables": 4}),
                                     ("sweep", {"batch": 300, "tables": 4, "iteration": 7}),
                                     ("large", {"batch": 70, "tables": 2, "variant": "bf16"})])
def test_round_trip_workloads(name, kw):
    wl = workloads.make(name, **kw)
    x = wl.x.numpy()
    eb = wl.eb.numpy()
    if wl.schedule:
        s = wl.schedule
        eb = o.scheduled_bounds(s["base"].numpy(), s["fn"], s["iteration"], s["m0"], s["phase_len"])
    buf, info, sym, ref, lens = o.compress(x, eb, want_internals=True)
    xh, sym2 = o.decompress(buf, *x.shape)
    assert (sym2 == sym).all()
    err = np.abs(x.astype(np.float64) - xh.astype(np.float64)).max(axis=(0, 2))
    assert (err <= eb.astype(np.float64)).all()
    assert info["total_bytes"] < x.nbytes


# ---------------------------------------------------------------- corruption
def test_corrupt_containers_rejected():
    wl = workloads.make("tiny", batch=128, tables=2)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    buf, info = o.compress(x, eb)
    B, T, D = x.shape
    assert o.decompress_rc(buf[:-1], B, T, D)[0] == o.ERR_CORRUPT
    bad = buf.copy(); bad[0] ^= 1
    assert o.decompress_rc(bad, B, T, D)[0] == o.ERR_CORRUPT
    assert o.decompress_rc(buf, B + 1, T, D)[0] == o.ERR_INVALID_ARG
    off_chunks = struct.unpack_from("<Q", buf.tobytes(), 104)[0]
    bad = buf.copy(); bad[off_chunks] ^= 1                 # a chunk length off by one
    assert o.decompress_rc(bad, B, T, D)[0] == o.ERR_CORRUPT
    bad = buf.copy(); bad[160 + 128] = 30                  # a code length beyond 24
    assert o.decompress_rc(bad, B, T, D)[0] == o.ERR_CORRUPT
    rng = np.random.default_rng(0)
    for _ in range(200):                                   # random flips: no crash
        bad = buf.copy()
        i = int(rng.integers(0, len(bad)))
        bad[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        assert o.decompress_rc(bad, B, T, D)[0] in (o.OK, o.ERR_CORRUPT, o.ERR_INVALID_ARG)
