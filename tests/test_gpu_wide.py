"""The wide alphabet on the GPU (radius 512: 1024 symbols, 16-bit codes in the
code scratch) against the oracle with the same radius ("Accelerating
Communication in Deep Learning Recommendation Model Training with Dual-Level
Adaptive Lossy Compression", §III-D quantization and Huffman encoders; the
paper fixes no radius).

Bar: containers byte-identical to the oracle's, reconstructions 0 ulp, on the
workloads (including the sigma = 1e-2 gradient case the alphabet is for),
every D, ragged batches, outliers past the wide bins, a Huffman code that hits
the 24-bit limit, windows, table modes, chunked buffers and bf16 input; a
container of the other alphabet is rejected."""
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
    c = ebc.Codec(0)
    c.set_radius(512)
    yield c
    c.close()


def _check(codec, x, eb, window=0, modes=None, bf16=False):
    codec.set_window(window)
    if modes is not None:
        codec.set_table_modes(modes)
    try:
        xd = torch.from_numpy(x).cuda()
        if bf16:
            xd = xd.to(torch.bfloat16)
        out, nb = codec.compress(xd, eb)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        n = int(nb.item())
        buf = out[:n].cpu().numpy()
        xh = codec.decompress(out, n, *x.shape)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        st = codec.stats()
    finally:
        codec.set_window(0)
        codec.set_table_modes(None)
    ref, info = oracle.compress(x, eb, window=window, modes=modes, radius=512)
    assert len(buf) == len(ref) and np.array_equal(buf, ref)
    xo, _ = oracle.decompress(ref, *x.shape)
    assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
    return info, st


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("fwd", {"batch": 2048}), ("bwd", {"batch": 4096}),
                                     ("bwd", {"variant": "s1e-2"}), ("fwd", {})])
def test_workloads_bit_exact(codec, name, kw):
    wl = workloads.make(name, **kw)
    _check(codec, wl.x.numpy(), wl.eb.numpy())


def _planted(B, T, D, seed):
    # duplicated rows, values over +-700 bins of eb (some past the wide bins), a few huge outliers
    rng = np.random.default_rng(seed)
    eb = (10.0 ** rng.uniform(-4, -2, T)).astype(np.float32)
    x = (rng.standard_normal((B, T, D)) * 250 * eb[None, :, None]).astype(np.float32)
    for t in range(T):
        src = rng.integers(0, max(B, 1), B)
        for b in np.nonzero(rng.uniform(size=B) < 0.5)[0]:
            if src[b] < b:
                x[b, t] = x[src[b], t]
    if x.size:
        k = max(1, x.size // 500)
        x.reshape(-1)[rng.integers(0, x.size, k)] = rng.standard_normal(k).astype(np.float32) * 1e4
    return x, eb


@pytest.mark.parametrize("D", [4, 8, 16, 64, 128, 512])
@pytest.mark.parametrize("B", [1, 1000, 5003])
def test_shapes_bit_exact(codec, B, D):
    x, eb = _planted(B, 3, D, seed=B * 7 + D)
    _check(codec, x, eb)


def test_length_limit(codec):
    # 2^24 codes with P(|q| = k) = 2^-k: the rarest bins would need codes longer than 24 bits
    rng = np.random.default_rng(12)
    B, D = 65536, 256
    eb = np.float32(1e-3)
    k = np.minimum(rng.geometric(0.5, (B, D)), 511)
    q = k * np.where(rng.uniform(size=(B, D)) < 0.5, -1, 1)
    x = (q * 2 * eb).astype(np.float32)[:, None, :]
    lens = oracle.compress(x, np.array([eb]), want_internals=True, radius=512)[4]
    assert lens.max() == 24
    _check(codec, x, np.array([eb], np.float32))


def test_degenerate_tables(codec):
    B, T, D = 700, 4, 32
    x = np.zeros((B, T, D), np.float32)                        # t=0: one symbol
    rng = np.random.default_rng(5)
    x[:, 1] = rng.standard_normal((B, D)).astype(np.float32)   # t=1: all distinct
    x[:, 2] = x[0, 2] + 0.0
    x[:, 2, 5] = np.float32(np.nan)                            # t=2: identical rows with a NaN
    x[::7, 3, :4] = [np.inf, -np.inf, np.float32(1e-42), -0.0]  # t=3: non-finite, subnormal, -0
    _check(codec, x, np.full(T, 1e-3, np.float32))


@pytest.mark.parametrize("window", [1, 64])
def test_windows(codec, window):
    wl = workloads.make("bwd", batch=3000, tables=6, variant="s1e-2")
    _check(codec, wl.x.numpy(), wl.eb.numpy(), window=window)


def test_table_modes_raw_codes_are_ten_bits(codec):
    wl = workloads.make("bwd", batch=2000, tables=8, variant="s1e-2")
    modes = np.array([0, 1, 2, 3, 0, 1, 2, 3], np.uint8)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), modes=modes)


def test_bf16_input(codec):
    wl = workloads.make("fwd", batch=1024, tables=4)
    x = wl.x.to(torch.bfloat16).float().numpy()
    _check(codec, x, wl.eb.numpy(), bf16=True)


@pytest.mark.parametrize("n", [2, 5])
def test_chunked(codec, n):
    wl = workloads.make("bwd", batch=2500, tables=5, variant="s1e-2")
    x, eb = wl.x.numpy(), wl.eb.numpy()
    out, offs = codec.compress_chunked(torch.from_numpy(x).cuda(), n, eb)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    o = offs.cpu().numpy()
    ref, roffs = oracle.compress_chunked(x, eb, n, radius=512)
    assert o.tolist() == roffs.tolist()
    assert np.array_equal(out[:int(o[-1])].cpu().numpy(), ref)
    xh = codec.decompress_chunked(out, int(o[-1]), offs, *x.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    assert np.array_equal(xh.cpu().numpy().view(np.uint32),
                          oracle.decompress_chunked(ref, roffs, *x.shape).view(np.uint32))


def test_fewer_outliers_than_the_narrow_alphabet(codec):
    wl = workloads.make("bwd", variant="s1e-2")
    info, st = _check(codec, wl.x.numpy(), wl.eb.numpy())
    _, narrow = oracle.compress(wl.x.numpy(), wl.eb.numpy())
    assert st["n_outlier"] == info["n_outlier"] and 3 * info["n_outlier"] < narrow["n_outlier"]


def test_other_alphabet_rejected(codec):
    wl = workloads.make("tiny")
    x = wl.x.cuda()
    wide, nw = codec.compress(x, wl.eb.numpy())
    narrow_codec = ebc.Codec(0)
    try:
        narrow, nn = narrow_codec.compress(x, wl.eb.numpy())
        torch.cuda.synchronize()
        for dec, buf, n in ((narrow_codec, wide, int(nw.item())), (codec, narrow, int(nn.item()))):
            xh = torch.empty_like(x)
            rc = ebc.ebc_decompress(dec.handle, ctypes.c_void_p(buf.data_ptr()), n, ctypes.c_void_p(xh.data_ptr()),
                                    *x.shape, None)
            assert rc == 0
            assert dec.last_error() == ebc.EBC_ERR_INVALID_ARG
        # both contexts still decode their own
        xh = narrow_codec.decompress(narrow, int(nn.item()), *x.shape)
        torch.cuda.synchronize()
        assert narrow_codec.last_error() == 0
    finally:
        narrow_codec.close()
    assert ebc.ebc_set_radius(codec.handle, 256) == ebc.EBC_ERR_INVALID_ARG
