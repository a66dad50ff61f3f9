"""Pins of the oracle's sliding-window vector LZ ("Accelerating Communication
in Deep Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-E "extended window size" and "fixed pattern length",
§IV-D Table VI): the reference of a vector is the nearest earlier vector of
its table within W rows with the same key, a match when the codes are equal;
references are one-byte distances and may chain."""
import numpy as np
import pytest

import oracle as o
import workloads


def _rows(pattern, D=4):
    # distinct, exactly representable rows (all in-range codes) keyed by a letter
    base = {c: np.arange(D, dtype=np.float32) * 0.25 + 0.125 * k for k, c in enumerate(sorted(set(pattern)))}
    x = np.stack([base[c] for c in pattern])[:, None, :].astype(np.float32)
    return x, np.array([1e-3], np.float32)


def _refs(buf, n_match):
    off_refs = int.from_bytes(bytes(buf[112:120]), "little")
    return list(bytes(buf[off_refs:off_refs + n_match]))


def test_hand_example_chains():
    x, eb = _rows("ABACA")
    # W = 2: row 2 -> row 0 (distance 2); row 4 -> row 2 (distance 2), itself a match
    buf, info, sym, ref, lens = o.compress(x, eb, want_internals=True, window=2)
    assert ref[0].tolist() == [0, 1, 0, 3, 2]
    assert info["n_match"] == 2
    assert int.from_bytes(bytes(buf[40:44]), "little") == 1      # one-byte references
    assert int.from_bytes(bytes(buf[44:48]), "little") == 2      # the window
    assert _refs(buf, 2) == [2, 2]
    xh, _ = o.decompress(buf, *x.shape)
    assert np.array_equal(xh, o.decompress(o.compress(x, eb)[0], *x.shape)[0])
    # W = 1: no A is adjacent to another A
    buf1, info1, _, ref1, _ = o.compress(x, eb, want_internals=True, window=1)
    assert info1["n_match"] == 0 and ref1[0].tolist() == [0, 1, 2, 3, 4]
    # whole batch: both later As name row 0
    _, _, _, ref0, _ = o.compress(x, eb, want_internals=True)
    assert ref0[0].tolist() == [0, 1, 0, 3, 0]


def test_long_chain_decodes():
    x, eb = _rows("A" * 300)
    buf, info, _, ref, _ = o.compress(x, eb, want_internals=True, window=1)
    assert info["n_match"] == 299 and ref[0, 1:].tolist() == list(range(299))
    xh, _ = o.decompress(buf, *x.shape)
    assert (xh == xh[0]).all()


def test_window_zero_is_the_default():
    wl = workloads.make("tiny")
    a, _ = o.compress(wl.x.numpy(), wl.eb.numpy())
    b, _ = o.compress(wl.x.numpy(), wl.eb.numpy(), window=0)
    assert np.array_equal(a, b)


def test_matches_grow_with_the_window_and_reconstruction_stays():
    wl = workloads.make("fwd", batch=1024)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    base = None
    last = -1
    for W in (1, 8, 32, 64, 128, 255):
        buf, info = o.compress(x, eb, window=W)
        assert info["n_match"] >= last
        last = info["n_match"]
        xh, _ = o.decompress(buf, *x.shape)
        if base is None:
            base = xh
        assert np.array_equal(xh.view(np.uint32), base.view(np.uint32))


def test_window_covering_the_batch_finds_every_duplicate():
    wl = workloads.make("tiny", batch=200)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    _, full = o.compress(x, eb)
    _, win = o.compress(x, eb, window=255)
    assert win["n_match"] == full["n_match"]


def test_bad_windows_and_distances():
    x, eb = _rows("ABACA")
    with pytest.raises(RuntimeError):
        o.compress(x, eb, window=256)
    buf, info = o.compress(x, eb, window=2)
    off_refs = int.from_bytes(bytes(buf[112:120]), "little")
    for bad in (0, 3):   # distance 0, or beyond the window
        b = buf.copy()
        b[off_refs] = bad
        rc, _, _ = o.decompress_rc(b, *x.shape)
        assert rc == o.ERR_CORRUPT
    b = buf.copy()
    b[44] = 0            # a whole-batch container cannot have one-byte references
    rc, _, _ = o.decompress_rc(b, *x.shape)
    assert rc == o.ERR_CORRUPT
