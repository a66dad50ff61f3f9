"""Parity of the CUDA codec with the CPU oracle, through the C ABI.

Bar: containers byte-identical to the oracle's (codes, dedup decisions,
codebooks, bitstreams, chunk index, layout) and reconstructions bit-identical
to the oracle decoder's (0 ulp), which also obey |x - xhat| <= eb_t on every
element.  Workloads: the five synthetic embedding-traffic configurations at
full size, plus shapes and edge cases that span several segments and ragged
tails.
"""
import ctypes

import numpy as np
import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import oracle
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(scope="module")
def codec():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    c = ebc.Codec(0)
    yield c
    c.close()


def gpu_roundtrip(codec, x_cpu, eb, x_dev=None):
    """(container bytes, xhat numpy, device error codes)."""
    x = x_dev if x_dev is not None else x_cpu.to("cuda")
    out, nb = codec.compress(x, eb)
    torch.cuda.synchronize()
    e1 = codec.last_error()
    n = int(nb.item())
    buf = out[:n].cpu().numpy()
    xh = codec.decompress(out, n, *x.shape)
    torch.cuda.synchronize()
    e2 = codec.last_error()
    return buf, xh.cpu().numpy(), (e1, e2)


def assert_parity(codec, x_cpu, eb, x_dev=None):
    x_np = x_cpu.numpy() if isinstance(x_cpu, torch.Tensor) else x_cpu
    eb = np.asarray(eb, np.float32)
    buf, xh, errs = gpu_roundtrip(codec, torch.from_numpy(x_np) if x_dev is None else None, eb, x_dev)
    assert errs == (0, 0)
    ref, info = oracle.compress(x_np, eb)
    assert len(buf) == len(ref), (len(buf), len(ref))
    if not np.array_equal(buf, ref):
        diff = np.nonzero(buf != ref)[0]
        raise AssertionError(f"{diff.size} bytes differ, first at {diff[:8]}")
    xo, _ = oracle.decompress(ref, *x_np.shape)
    assert np.array_equal(xh.view(np.uint32), xo.view(np.uint32))
    # the bound, element by element (outliers are exact)
    err = np.abs(x_np.astype(np.float64) - xh.astype(np.float64))
    finite = np.isfinite(x_np)
    lim = np.broadcast_to(eb.astype(np.float64)[None, :, None], x_np.shape)
    assert (err[finite] <= lim[finite]).all()
    return info


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("fwd", {}),
    ("bwd", {}),
    ("large", {"batch": 2048}),
    ("large", {"batch": 2048, "variant": "bf16"}),
])
def test_workloads_bit_exact(codec, name, kw):
    wl = workloads.make(name, **kw)
    info = assert_parity(codec, wl.x, wl.eb.numpy())
    assert info["total_bytes"] < wl.nbytes


@pytest.mark.parametrize("first", [0, 20, 40, 60, 80])
def test_sweep_all_iterations_with_schedule(codec, first):
    """The iteration-wise sweep, all 100 iterations (20 per test): each batch is
    generated on the device, compressed with the context's decayed bounds
    (eb = None) and compared byte for byte with the oracle's container; every
    reconstruction meets its bound, and every tenth is compared with the oracle
    decoder bit for bit."""
    for it in range(first, first + 20):
        wl = workloads.make("sweep", iteration=it, device="cuda")
        s = wl.schedule
        base = s["base"].numpy()
        codec.set_error_bounds(base, s["iteration"], s["fn"], s["m0"], s["phase_len"], s["n_steps"])
        want = oracle.scheduled_bounds(base, s["fn"], s["iteration"], s["m0"], s["phase_len"], s["n_steps"])
        assert np.array_equal(codec.error_bounds(base.size), want)
        out, nb = codec.compress(wl.x, None)
        torch.cuda.synchronize()
        assert codec.last_error() == 0, it
        n = int(nb.item())
        x_np = wl.x.cpu().numpy()
        ref, _ = oracle.compress(x_np, want)
        got = out[:n].cpu().numpy()
        assert n == len(ref) and np.array_equal(got, ref), f"iteration {it}: container differs"
        xh = codec.decompress(out, n, *wl.shape)
        torch.cuda.synchronize()
        assert codec.last_error() == 0, it
        err = (wl.x.double() - xh.double()).abs().amax(dim=(0, 2)).cpu().numpy()
        assert (err <= want.astype(np.float64)).all(), f"iteration {it}: bound violated"
        if it % 10 == 0:
            xo, _ = oracle.decompress(ref, *wl.shape)
            assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32)), it


@pytest.mark.parametrize("fn", ["none", "linear", "stepwise", "drop", "log"])
def test_schedule_matches_oracle(codec, fn):
    base = np.array([1e-3, 2.5e-2, 7e-4, 0.3], np.float32)
    for it in [0, 1, 5, 17, 39, 40, 100]:
        codec.set_error_bounds(base, it, fn, 3.0, 40, 4)
        assert np.array_equal(codec.error_bounds(4), oracle.scheduled_bounds(base, fn, it, 3.0, 40, 4))


def _planted(B, T, D, seed, dup=0.5, outl=0.002, scale=0.05):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((B, T, D)) * scale).astype(np.float32)
    for t in range(T):
        src = rng.integers(0, max(B, 1), B)
        m = rng.uniform(size=B) < dup
        for b in np.nonzero(m)[0]:
            if src[b] < b:
                x[b, t] = x[src[b], t]
    if x.size:
        k = max(1, int(x.size * outl))
        x.reshape(-1)[rng.integers(0, x.size, k)] = rng.standard_normal(k).astype(np.float32) * 1e4
    eb = (10.0 ** rng.uniform(-4, -2, T)).astype(np.float32)
    return x, eb


@pytest.mark.parametrize("D", [4, 8, 16, 32, 64, 128, 256, 512])
@pytest.mark.parametrize("B", [1, 33, 1000, 5003])
def test_shapes_bit_exact(codec, B, D):
    T = 3
    x, eb = _planted(B, T, D, seed=B * 131 + D)
    assert_parity(codec, x, eb)


def test_empty_inputs(codec):
    for B, T, D in [(0, 3, 16), (5, 0, 128), (0, 0, 4)]:
        x = np.zeros((B, T, D), np.float32)
        eb = np.full((T,), 1e-3, np.float32)
        if B * T * D == 0:
            xd = torch.zeros((B, T, D), dtype=torch.float32, device="cuda")
            out, nb = codec.compress(xd, eb)
            torch.cuda.synchronize()
            assert codec.last_error() == 0
            n = int(nb.item())
            ref, _ = oracle.compress(x, eb)
            assert np.array_equal(out[:n].cpu().numpy(), ref)
            xh = codec.decompress(out, n, B, T, D)
            torch.cuda.synchronize()
            assert codec.last_error() == 0 and xh.numel() == 0


def test_degenerate_tables(codec):
    B, T, D = 700, 5, 32
    x = np.zeros((B, T, D), np.float32)                    # t=0: one symbol, all rows equal
    rng = np.random.default_rng(9)
    x[:, 1] = rng.standard_normal((B, D)).astype(np.float32)   # t=1: all distinct, wide values
    x[:, 2] = x[0, 2] + 0.0                                 # t=2: identical rows
    x[:, 2, 5] = np.float32(np.nan)
    x[::7, 3, :4] = [np.inf, -np.inf, np.float32(1e-42), -0.0]  # t=3: non-finite, subnormal, -0
    x.view(np.uint32)[3, 3, 9] = 0x7FC01234                # NaN payload
    # t=4: geometric histogram across many bins, forcing long codes
    eb4 = np.float32(1e-3)
    q = np.minimum(rng.geometric(0.35, (B, D)), 120) * np.where(rng.uniform(size=(B, D)) < 0.5, -1, 1)
    x[:, 4] = (q * 2 * eb4).astype(np.float32)
    eb = np.array([1e-3, 1e-3, 1e-3, 1e-3, eb4], np.float32)
    assert_parity(codec, x, eb)


def test_half_bin_ties(codec):
    eb = np.float32(1e-3)
    k = np.arange(-130, 131, dtype=np.float64)
    vals = np.concatenate([(k + 0.5) * 2 * float(eb), k * 2 * float(eb)]).astype(np.float32)
    D = 16
    B = -(-vals.size // D)
    x = np.zeros(B * D, np.float32)
    x[: vals.size] = vals
    assert_parity(codec, x.reshape(B, 1, D), np.array([eb], np.float32))


def test_repeat_calls_deterministic_and_growth(codec):
    x1, eb1 = _planted(3000, 4, 64, seed=1)
    x2, eb2 = _planted(20000, 7, 128, seed=2)
    bufs = []
    for x, eb in [(x1, eb1), (x2, eb2), (x1, eb1), (x2, eb2)]:
        buf, xh, errs = gpu_roundtrip(codec, torch.from_numpy(x), eb)
        assert errs == (0, 0)
        bufs.append(buf)
    assert np.array_equal(bufs[0], bufs[2]) and np.array_equal(bufs[1], bufs[3])


def test_two_contexts_two_streams():
    x1, eb1 = _planted(4000, 5, 128, seed=3)
    x2, eb2 = _planted(4000, 5, 32, seed=4)
    c1, c2 = ebc.Codec(0), ebc.Codec(0)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    d1, d2 = torch.from_numpy(x1).cuda(), torch.from_numpy(x2).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        o1, n1 = c1.compress(d1, eb1, stream=s1)
    with torch.cuda.stream(s2):
        o2, n2 = c2.compress(d2, eb2, stream=s2)
    torch.cuda.synchronize()
    assert c1.last_error() == 0 and c2.last_error() == 0
    r1, _ = oracle.compress(x1, eb1)
    r2, _ = oracle.compress(x2, eb2)
    assert np.array_equal(o1[: int(n1.item())].cpu().numpy(), r1)
    assert np.array_equal(o2[: int(n2.item())].cpu().numpy(), r2)
    c1.close()
    c2.close()


def test_host_buffer_calls(codec):
    wl = workloads.make("fwd", batch=1024)
    xh_pinned = wl.x.pin_memory()
    buf, n = codec.compress_host(xh_pinned, wl.eb.numpy())
    ref, _ = oracle.compress(wl.x.numpy(), wl.eb.numpy())
    assert n == len(ref) and np.array_equal(buf[:n].numpy(), ref)
    out = codec.decompress_host(buf, n, *wl.shape)
    xo, _ = oracle.decompress(ref, *wl.shape)
    assert np.array_equal(out.numpy().view(np.uint32), xo.view(np.uint32))


def test_capacity_too_small(codec):
    wl = workloads.make("tiny")
    x = wl.x.cuda()
    eb = wl.eb.numpy()
    ref, _ = oracle.compress(wl.x.numpy(), eb)
    B, T, D = wl.shape
    # below the fixed-size head: rejected before any launch
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(ebc.EbcError) as e:
        codec.compress_into(x, eb, small, nb)
    assert e.value.code == ebc.EBC_ERR_CAPACITY
    # room for the head only: the kernels report the required size
    cap = len(ref) - 100
    out = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    codec.compress_into(x, eb, out, nb)
    torch.cuda.synchronize()
    assert codec.last_error() == ebc.EBC_ERR_CAPACITY
    assert int(nb.item()) == len(ref)
    # the context stays usable
    assert_parity(codec, wl.x, eb)


def test_bad_arguments(codec):
    x = torch.zeros((4, 2, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(ebc.EbcError):
        codec.compress(x, np.array([0.0, 1e-3], np.float32))
    with pytest.raises(ebc.EbcError):
        codec.compress(x, np.array([np.nan, 1e-3], np.float32))
    with pytest.raises(ebc.EbcError):
        codec.compress(torch.zeros((4, 2, 24), dtype=torch.float32, device="cuda"), np.ones(2, np.float32))
    with pytest.raises(ebc.EbcError):
        codec.compress(x, None)   # no schedule for T = 2 yet


def _decode_rc(codec, buf, shape):
    d = torch.from_numpy(np.ascontiguousarray(buf)).cuda()
    xh = torch.empty(shape, dtype=torch.float32, device="cuda")
    codec.decompress_into(d, len(buf), xh)
    torch.cuda.synchronize()
    return codec.last_error(), xh


def _corruption_cases(ref, rng, n_random, tables=2):
    """Single-bit flips: a few in every section of the container, then random ones."""
    h = lambda o: int(np.frombuffer(ref[o:o + 8].tobytes(), np.uint64)[0])
    off_seg, off_bitmap, off_chunks, off_refs, off_bits = h(88), h(96), h(104), h(112), h(120)
    sections = [(0, 144), (144, off_seg), (off_seg, off_bitmap), (off_bitmap, off_chunks),
                (off_chunks, off_refs), (off_refs, off_bits), (off_bits, len(ref))]
    # the counts of each table record (literals, matches, outliers) and the header's counts
    fields = [64, 48, 56, 72, 80] + [144 + k * 272 + f for k in range(tables) for f in (4, 8, 12)]
    cases = [(i, b) for i in fields for b in (0, 1, 5)]
    for lo, hi in sections:
        if hi > lo:
            cases += [(int(rng.integers(lo, hi)), int(rng.integers(0, 8))) for _ in range(6)]
    cases += [(int(rng.integers(0, len(ref))), int(rng.integers(0, 8))) for _ in range(n_random)]
    return cases


@pytest.mark.parametrize("window", [0, 16])
def test_corrupt_containers(codec, window):
    """The GPU decoder rejects exactly the containers the oracle's decoder rejects,
    with the same code, and when both accept one, their reconstructions agree bit
    for bit; the context keeps working."""
    wl = workloads.make("tiny", batch=256, tables=2)
    x, eb = wl.x.numpy().copy(), wl.eb.numpy()
    x[3, 1, 5] = np.float32(7.5)          # outliers, so that the outlier counts are checked too
    x[200, 0, 0] = np.float32(-3.25)
    ref, info = oracle.compress(x, eb, window=window)
    assert info["n_outlier"] >= 2 and info["n_match"] > 0
    shape = x.shape
    codec.set_window(window)
    try:
        assert _decode_rc(codec, ref, shape)[0] == 0
        assert _decode_rc(codec, ref[:-1], shape)[0] == ebc.EBC_ERR_CORRUPT
        assert _decode_rc(codec, ref, (shape[0] + 1,) + shape[1:])[0] == ebc.EBC_ERR_INVALID_ARG
        rng = np.random.default_rng(window)
        n_both_ok = 0
        for i, bit in _corruption_cases(ref, rng, 120):
            bad = ref.copy()
            bad[i] ^= np.uint8(1 << bit)
            rc_o, xo, _ = oracle.decompress_rc(bad, *shape)
            rc_g, xg = _decode_rc(codec, bad, shape)
            assert rc_g == rc_o, (i, bit, rc_g, rc_o)
            if rc_o == oracle.OK:
                n_both_ok += 1
                assert np.array_equal(xg.cpu().numpy().view(np.uint32), xo.view(np.uint32)), (i, bit)
        assert n_both_ok > 0
        # still usable
        rc, xg = _decode_rc(codec, ref, shape)
        assert rc == 0
        assert np.array_equal(xg.cpu().numpy().view(np.uint32), oracle.decompress(ref, *shape)[0].view(np.uint32))
    finally:
        codec.set_window(0)


@pytest.mark.parametrize("window", [0, 16])
def test_corrupt_containers_shares(codec, window):
    """As test_corrupt_containers, with rows of 128 codes (a chunk per row), where every decode CTA
    takes an equal share of its table's chunks (far more CTAs than segment groups): the GPU rejects
    exactly what the oracle rejects, with the same code, and agrees bit for bit when both accept.
    Flips in the segment records and chunk table reach the shares' range search and start bits."""
    wl = workloads.make("fwd", batch=512, tables=3)
    x, eb = wl.x.numpy().copy(), wl.eb.numpy()
    x[3, 1, 5] = np.float32(1e3)           # outliers
    x[200, 0, 0] = np.float32(-1e3)
    ref, info = oracle.compress(x, eb, window=window)
    assert info["n_outlier"] >= 2 and info["n_match"] > 0 and info["n_literal"] > 0
    shape = x.shape
    codec.set_window(window)
    try:
        assert _decode_rc(codec, ref, shape)[0] == 0
        h = lambda o: int(np.frombuffer(ref[o:o + 8].tobytes(), np.uint64)[0])
        rng = np.random.default_rng(100 + window)
        cases = _corruption_cases(ref, rng, 60, tables=3)
        # more flips in the segment records (chunk bases, word offsets) and the chunk table
        cases += [(int(rng.integers(h(88), h(96))), int(rng.integers(0, 8))) for _ in range(40)]
        cases += [(int(rng.integers(h(104), h(112))), int(rng.integers(0, 8))) for _ in range(20)]
        n_both_ok = 0
        for i, bit in cases:
            bad = ref.copy()
            bad[i] ^= np.uint8(1 << bit)
            rc_o, xo, _ = oracle.decompress_rc(bad, *shape)
            rc_g, xg = _decode_rc(codec, bad, shape)
            assert rc_g == rc_o, (i, bit, rc_g, rc_o)
            if rc_o == oracle.OK:
                n_both_ok += 1
                assert np.array_equal(xg.cpu().numpy().view(np.uint32), xo.view(np.uint32)), (i, bit)
        assert n_both_ok > 0
        rc, xg = _decode_rc(codec, ref, shape)
        assert rc == 0
        assert np.array_equal(xg.cpu().numpy().view(np.uint32), oracle.decompress(ref, *shape)[0].view(np.uint32))
    finally:
        codec.set_window(0)


def test_full_size_large_batch(codec):
    """[65536, 26, 256] (1.7 GB) and its bf16-cast variant, whole container vs the oracle."""
    for variant in (None, "bf16"):
        wl = workloads.make("large", device="cuda", variant=variant)
        x_cpu = wl.x.cpu()
        assert_parity(codec, x_cpu.numpy(), wl.eb.numpy(), x_dev=wl.x)
        del wl, x_cpu
        torch.cuda.empty_cache()
