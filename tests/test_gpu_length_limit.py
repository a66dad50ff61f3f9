"""The Huffman length limit on the GPU, against the oracle.

The code of a unit is built from its literal-code histogram; when the
two-queue construction gives a code longer than 24 bits, every nonzero count
becomes max(1, count >> 1) and the code is rebuilt, until it fits (the
length-limited reading of the Huffman encoder of "Accelerating Communication in
Deep Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-D).  Ordinary embedding batches never need it, so these
tables are built to: the literal codes of one table take k distinct bins with
Fibonacci counts F_1 .. F_k, the weights whose Huffman tree is a chain of depth
k - 1.  The test first asks the oracle how many halving rounds the literal
histogram needs (at least one), then requires the GPU container to be
byte-identical to the oracle's and its reconstruction bit-identical to the
oracle decoder's, for both alphabets and for both ways the GPU lays out the
segment offsets (inside the code-building kernel for units of at most 256
segments, by the separate layout kernel above that).
"""
import numpy as np
import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def fibonacci_table(nbins: int, D: int, seed: int, spread: int = 1):
    """One table [B, 1, D] whose codes take nbins bins (spread apart) with
    Fibonacci counts, shuffled over the rows; eb = 2^-10 so every value sits
    exactly on its bin."""
    f = [1, 1]
    while len(f) < nbins:
        f.append(f[-1] + f[-2])
    rng = np.random.default_rng(seed)
    qs = (np.arange(nbins) - nbins // 2) * spread
    codes = np.repeat(qs, f)
    codes = np.concatenate([codes, np.full((-codes.size) % D, qs[-1])])
    rng.shuffle(codes)
    eb = np.float32(2.0 ** -10)
    x = (codes.astype(np.float64) * 2.0 * float(eb)).astype(np.float32).reshape(-1, 1, D)
    return x, np.array([eb], np.float32)


def halving_rounds(x, eb, radius):
    """Halving rounds the oracle's code of table 0 needed, from its literal histogram."""
    _, _, sym, ref, lens = oracle.compress(x, eb, want_internals=True, radius=radius)
    lit = ref[0] == np.arange(x.shape[0])
    hist = np.bincount(sym[0][lit].reshape(-1).astype(np.int64), minlength=2 * radius)
    ln, rounds = oracle.huffman_lengths(hist, symbols=2 * radius)
    assert np.array_equal(ln, lens[0])
    return rounds, int(ln.max())


@pytest.fixture()
def codec():
    c = ebc.Codec(0)
    yield c
    c.close()


@pytest.mark.parametrize("radius,nbins,D,spread", [
    (128, 30, 128, 1),    # 17,019 rows: 266 segments, offsets by the layout kernel
    (128, 30, 512, 1),    # 4,255 rows: 133 segments, offsets inside the code build
    (128, 33, 256, 3),    # 3 x more weight: 3 halving rounds
    (512, 31, 128, 25),   # wide alphabet, bins 25 apart (codes up to +-375)
    (512, 32, 64, 30),    # wide alphabet, 89,108 rows, longest code exactly 24 after halving
])
def test_length_limit_halving_bit_exact(codec, radius, nbins, D, spread):
    x, eb = fibonacci_table(nbins, D, seed=nbins * 7 + D, spread=spread)
    rounds, maxlen = halving_rounds(x, eb, radius)
    assert rounds >= 1 and maxlen <= oracle.LMAX
    codec.set_radius(radius)
    xd = torch.from_numpy(x).cuda()
    out, nb = codec.compress(xd, eb)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    n = int(nb.item())
    ref, _ = oracle.compress(x, eb, radius=radius)
    got = out[:n].cpu().numpy()
    assert n == len(ref)
    if not np.array_equal(got, ref):
        diff = np.nonzero(got != ref)[0]
        raise AssertionError(f"{diff.size} bytes differ, first at {diff[:8]}")
    xh = codec.decompress(out, n, *x.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    xo, _ = oracle.decompress(ref, *x.shape)
    assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
    assert np.array_equal(xo, x)   # every value sits on its bin


def test_length_limit_among_ordinary_tables(codec):
    """A halving table between two ordinary tables of the same batch: only its
    own code is rebuilt."""
    xf, ebf = fibonacci_table(30, 128, seed=5)
    B = xf.shape[0]
    rng = np.random.default_rng(6)
    x = np.empty((B, 3, 128), np.float32)
    x[:, 0] = rng.uniform(-0.05, 0.05, (B, 128)).astype(np.float32)
    x[:, 1] = xf[:, 0]
    x[:, 2] = x[rng.integers(0, B, B), 0]
    eb = np.array([1e-3, ebf[0], 1e-3], np.float32)
    assert halving_rounds(xf, ebf, 128)[0] >= 1
    xd = torch.from_numpy(x).cuda()
    out, nb = codec.compress(xd, eb)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    n = int(nb.item())
    ref, _ = oracle.compress(x, eb)
    assert n == len(ref) and np.array_equal(out[:n].cpu().numpy(), ref)
    xh = codec.decompress(out, n, *x.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    xo, _ = oracle.decompress(ref, *x.shape)
    assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
