"""Sliding-window vector LZ on the GPU against the oracle ("Accelerating
Communication in Deep Learning Recommendation Model Training with Dual-Level
Adaptive Lossy Compression", §III-E "extended window size", §IV-D Table VI).

Bar: containers byte-identical to the oracle's with the same window,
reconstructions 0 ulp (chained references resolved on the GPU)."""
import numpy as np
import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import oracle
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(scope="module")
def codec():
    c = ebc.Codec(0)
    yield c
    c.close()


def _check(codec, x, eb, window, modes=None):
    codec.set_window(window)
    if modes is not None:
        codec.set_table_modes(modes)
    try:
        xd = torch.from_numpy(x).cuda()
        out, nb = codec.compress(xd, eb)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        n = int(nb.item())
        buf = out[:n].cpu().numpy()
        xh = codec.decompress(out, n, *x.shape)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
    finally:
        codec.set_window(0)
        codec.set_table_modes(None)
    ref, info = oracle.compress(x, eb, window=window, modes=modes)
    assert len(buf) == len(ref) and np.array_equal(buf, ref)
    xo, _ = oracle.decompress(ref, *x.shape)
    assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
    return info


@pytest.mark.parametrize("window", [1, 32, 64, 128, 255])
@pytest.mark.parametrize("name,kw", [("tiny", {}), ("fwd", {}), ("bwd", {"batch": 4096})])
def test_windows_bit_exact(codec, window, name, kw):
    wl = workloads.make(name, **kw)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), window)


@pytest.mark.parametrize("shape", [(1000, 3, 4), (777, 5, 64), (300, 2, 512)])
def test_window_shapes_and_long_chains(codec, shape):
    B, T, D = shape
    rng = np.random.default_rng(B)
    pool = rng.uniform(-0.05, 0.05, size=(3, T, D)).astype(np.float32)
    # a few vectors repeated in long runs: chains of hundreds of references
    x = np.ascontiguousarray(pool[(np.arange(B) // 97) % 3])
    eb = np.full(T, 1e-3, np.float32)
    info = _check(codec, x, eb, 1)
    assert info["n_match"] >= B * T - 40 * T


def test_window_with_modes(codec):
    wl = workloads.make("fwd", batch=2048)
    T = wl.x.shape[1]
    modes = np.random.default_rng(3).integers(0, 4, size=T).astype(np.uint8)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), 64, modes)


def test_window_ratio_grows(codec):
    wl = workloads.make("fwd")
    x, eb = wl.x.cuda(), wl.eb.numpy()
    sizes = []
    for w in (32, 64, 128, 255):
        codec.set_window(w)
        out, nb = codec.compress(x, eb)
        torch.cuda.synchronize()
        sizes.append(int(nb.item()))
    codec.set_window(0)
    assert sizes == sorted(sizes, reverse=True)


def test_bad_window_and_corrupt_distance(codec):
    with pytest.raises(ebc.EbcError):
        codec.set_window(256)
    wl = workloads.make("tiny")
    x = wl.x.numpy()
    ref, info = oracle.compress(x, wl.eb.numpy(), window=32)
    assert info["n_match"] > 0
    off_refs = int.from_bytes(bytes(ref[112:120]), "little")
    bad = ref.copy()
    bad[off_refs] = 0
    d = torch.from_numpy(bad).cuda()
    codec.decompress(d, len(bad), *x.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == ebc.EBC_ERR_CORRUPT
    # the context stays usable
    good = torch.from_numpy(ref).cuda()
    xh = codec.decompress(good, len(ref), *x.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
