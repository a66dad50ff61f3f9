"""Pins of the oracle's chunked sending buffer ("Accelerating Communication in
Deep Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-E "Buffer Optimization", Fig. 7; §IV-D, Fig. 15): the
batch is split equally into one slice per destination rank, each slice is
compressed as a container of its own, and the containers lie back to back in
one buffer.  Pinned against numpy's array_split (the slice boundaries), hand
examples of the dedup scope (a slice never refers into another), the error
bound, and the one-slice case, which must be the plain container."""
import numpy as np
import pytest

import oracle as o
import workloads


def _u64(buf, off):
    return int.from_bytes(bytes(buf[off:off + 8]), "little")


@pytest.mark.parametrize("B,n", [(10, 1), (10, 3), (10, 4), (8192, 16), (7, 7), (3, 5), (0, 2), (65537, 2)])
def test_slices_are_array_split(B, n):
    want = [(int(a[0]), int(a[-1]) + 1) if a.size else None for a in np.array_split(np.arange(B), n)]
    got = o.chunk_rows(B, n)
    assert len(got) == n
    for (b0, b1), w in zip(got, want):
        if w is None:
            assert b0 == b1
        else:
            assert (b0, b1) == w
    assert got[0][0] == 0 and got[-1][1] == B
    assert all(got[r][1] == got[r + 1][0] for r in range(n - 1))


def test_one_chunk_is_the_plain_container():
    wl = workloads.make("tiny")
    x, eb = wl.x.numpy(), wl.eb.numpy()
    buf, offs = o.compress_chunked(x, eb, 1)
    plain, _ = o.compress(x, eb)
    assert np.array_equal(buf, plain)
    assert offs.tolist() == [0, plain.size]


def _rows(pattern, D=4):
    base = {c: np.arange(D, dtype=np.float32) * 0.25 + 0.125 * k for k, c in enumerate(sorted(set(pattern)))}
    x = np.stack([base[c] for c in pattern])[:, None, :].astype(np.float32)
    return x, np.array([1e-3], np.float32)


def test_hand_example_dedup_stays_inside_a_slice():
    # "AABA" in two slices "AA" | "BA": the first slice has one match (row 1 -> row 0); the
    # second has none, its A's only earlier copy lying in the other slice
    x, eb = _rows("AABA")
    buf, offs = o.compress_chunked(x, eb, 2)
    c0 = buf[int(offs[0]):int(offs[1])]
    c1 = buf[int(offs[1]):int(offs[2])]
    assert (_u64(c0, 8), _u64(c0, 48), _u64(c0, 56)) == (2, 1, 1)    # B, literals, matches
    assert (_u64(c1, 8), _u64(c1, 48), _u64(c1, 56)) == (2, 2, 0)
    _, whole = o.compress(x, eb)
    assert whole["n_match"] == 2
    # a window is counted inside the slice too: "ABAB" | "ABAB" with W = 2
    x, eb = _rows("ABABABAB")
    buf, offs = o.compress_chunked(x, eb, 2, window=2)
    for r in range(2):
        c = buf[int(offs[r]):int(offs[r + 1])]
        assert _u64(c, 56) == 2 and int.from_bytes(bytes(c[44:48]), "little") == 2


def test_containers_are_self_contained_and_aligned():
    wl = workloads.make("tiny", batch=333)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    buf, offs = o.compress_chunked(x, eb, 5)
    assert offs[0] == 0 and offs[-1] == buf.size
    for r, (b0, b1) in enumerate(o.chunk_rows(333, 5)):
        c = buf[int(offs[r]):int(offs[r + 1])]
        assert int(offs[r]) % 16 == 0
        assert _u64(c, 8) == b1 - b0                # the slice's rows
        assert _u64(c, 128) == c.size               # its own total size
        alone, _ = o.compress(x[b0:b1], eb)
        assert np.array_equal(c, alone)


def test_error_bound_and_duplicate_rows_after_the_round_trip():
    wl = workloads.make("fwd", batch=1000, tables=4)
    x, eb = wl.x.numpy(), wl.eb.numpy()
    for n in (1, 3, 8):
        buf, offs = o.compress_chunked(x, eb, n)
        xh = o.decompress_chunked(buf, offs, *x.shape)
        err = np.abs(x.astype(np.float64) - xh.astype(np.float64))
        assert (err <= eb.astype(np.float64)[None, :, None]).all()
        # equal input rows inside one slice come back equal
        for b0, b1 in o.chunk_rows(x.shape[0], n):
            for t in range(x.shape[1]):
                rows = x[b0:b1, t]
                _, first, inv = np.unique(rows, axis=0, return_index=True, return_inverse=True)
                inv = inv.reshape(-1)
                assert np.array_equal(xh[b0:b1, t], xh[b0:b1, t][first[inv]])


def test_empty_slices():
    x, eb = _rows("AB")
    buf, offs = o.compress_chunked(x, eb, 4)      # slices of 1, 1, 0 and 0 rows
    sizes = np.diff(offs.astype(np.int64))
    assert (sizes > 0).all()
    for r, (b0, b1) in enumerate(o.chunk_rows(2, 4)):
        assert _u64(buf[int(offs[r]):int(offs[r + 1])], 8) == b1 - b0
    xh = o.decompress_chunked(buf, offs, 2, 1, 4)
    assert np.array_equal(xh, o.decompress(o.compress(x, eb)[0], 2, 1, 4)[0])


def test_columns_of_a_wider_output():
    # three senders with 2, 3 and 1 tables fill the columns of one [B, 6, D] output
    wl = workloads.make("tiny", batch=100)
    x, eb = wl.x.numpy(), wl.eb.numpy()          # [100, 4, 16]
    parts = [x[:, 0:2], x[:, 1:4], x[:, 3:4]]
    out = np.full((100, 6, 16), np.float32(7.0))
    col = 0
    for p, e in zip(parts, (eb[0:2], eb[1:4], eb[3:4])):
        p = np.ascontiguousarray(p)
        buf, _ = o.compress(p, e)
        o.decompress_columns(buf, 100, p.shape[1], 16, 6, col, out=out)
        assert np.array_equal(out[:, col:col + p.shape[1]], o.decompress(buf, *p.shape)[0])
        col += p.shape[1]
    assert col == 6
    with pytest.raises(ValueError):
        o.decompress_columns(buf, 100, 1, 16, 6, 6)
