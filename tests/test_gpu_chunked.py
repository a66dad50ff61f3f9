"""Chunked sending buffer on the GPU against the oracle ("Accelerating
Communication in Deep Learning Recommendation Model Training with Dual-Level
Adaptive Lossy Compression", §III-E "Buffer Optimization", Fig. 7; §IV-D,
Fig. 15): one self-contained container per batch slice, all written by one
pass of the kernels, and all decoded by one pass.

Bar: the buffer and the container boundaries byte-identical to the oracle's
(whose container r is its plain compress of slice r), reconstructions 0 ulp,
for ragged and empty slices, slices that start off a 16-byte boundary of the
code scratch (D = 4, 8), the folded and the tiled segment layouts, both
reference widths, windows, table modes and bf16 input; bad boundaries and
mismatched containers are rejected."""
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
    yield c
    c.close()


def _gpu(codec, x, eb, n, window=0, modes=None, bf16=False):
    codec.set_window(window)
    if modes is not None:
        codec.set_table_modes(modes)
    try:
        xd = torch.from_numpy(x).cuda()
        if bf16:
            xd = xd.to(torch.bfloat16)
        out, offs = codec.compress_chunked(xd, n, eb)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        o = offs.cpu().numpy().astype(np.uint64)
        total = int(o[-1])
        xh = codec.decompress_chunked(out, total, offs, *x.shape)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
    finally:
        codec.set_window(0)
        codec.set_table_modes(None)
    return out[:total].cpu().numpy(), o, xh.cpu().numpy()


def _check(codec, x, eb, n, window=0, modes=None):
    buf, offs, xh = _gpu(codec, x, eb, n, window, modes)
    ref, roffs = oracle.compress_chunked(x, eb, n, window=window, modes=modes)
    assert offs.tolist() == roffs.tolist()
    assert len(buf) == len(ref) and np.array_equal(buf, ref)
    xo = oracle.decompress_chunked(ref, roffs, *x.shape)
    assert np.array_equal(xh.view(np.uint32), xo.view(np.uint32))
    return buf, offs


@pytest.mark.parametrize("n", [1, 2, 3, 5, 16])
def test_tiny_bit_exact(codec, n):
    wl = workloads.make("tiny")
    _check(codec, wl.x.numpy(), wl.eb.numpy(), n)


@pytest.mark.parametrize("n", [3, 8])
def test_forward_workload_bit_exact(codec, n):
    wl = workloads.make("fwd", batch=1000, tables=6)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), n)


def test_full_forward_workload_eight_slices(codec):
    wl = workloads.make("fwd")
    _check(codec, wl.x.numpy(), wl.eb.numpy(), 8)


def _dup_rows(B, T, D, seed, pool=7):
    rng = np.random.default_rng(seed)
    p = rng.uniform(-0.05, 0.05, size=(pool, T, D)).astype(np.float32)
    return np.ascontiguousarray(p[rng.integers(0, pool, size=B)]), np.full(T, 1e-3, np.float32)


@pytest.mark.parametrize("shape,n", [((77, 3, 4), 5), ((1001, 2, 8), 7), ((130, 3, 4), 3), ((4099, 2, 16), 6)])
def test_unaligned_slice_starts(codec, shape, n):
    # slices start at rows whose codes are not 16-byte aligned in the table-major scratch
    x, eb = _dup_rows(*shape, seed=shape[0])
    _check(codec, x, eb, n)


@pytest.mark.parametrize("B,n", [(3, 5), (1, 4), (0, 4), (0, 1), (9, 9)])
def test_empty_slices(codec, B, n):
    x, eb = _dup_rows(B, 2, 16, seed=B + 100)
    buf, offs = _check(codec, x, eb, n)
    assert (np.diff(offs.astype(np.int64)) > 0).all()


def test_tiled_layout_long_slices(codec):
    # 16500 rows per slice at D = 128: 258 segments per table, past the folded layout's 256
    x, eb = _dup_rows(33000, 2, 128, seed=5, pool=4000)
    _check(codec, x, eb, 2)


def test_reference_widths_differ_between_slices(codec):
    # slices of 65537 and 65536 rows: four-byte references in the first, two-byte in the second
    x, eb = _dup_rows(131073, 1, 4, seed=9, pool=50000)
    buf, offs = _check(codec, x, eb, 2)
    assert int.from_bytes(bytes(buf[40:44]), "little") == 4
    second = buf[int(offs[1]):]
    assert int.from_bytes(bytes(second[40:44]), "little") == 2


@pytest.mark.parametrize("window", [1, 64, 255])
def test_windows(codec, window):
    wl = workloads.make("fwd", batch=2000, tables=4)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), 4, window=window)


def test_table_modes(codec):
    wl = workloads.make("fwd", batch=1500, tables=8)
    modes = np.array([0, 1, 2, 3, 0, 1, 2, 3], np.uint8)
    _check(codec, wl.x.numpy(), wl.eb.numpy(), 3, modes=modes)


def test_bf16_input(codec):
    wl = workloads.make("fwd", batch=1024, tables=4)
    x = wl.x.to(torch.bfloat16).float().numpy()   # the values bf16 holds, exactly
    buf, offs, xh = _gpu(codec, x, wl.eb.numpy(), 5, bf16=True)
    ref, roffs = oracle.compress_chunked(x, wl.eb.numpy(), 5)
    assert offs.tolist() == roffs.tolist() and np.array_equal(buf, ref)


def test_each_container_is_the_plain_container_of_its_slice(codec):
    wl = workloads.make("tiny", batch=300)
    x = wl.x.cuda()
    out, offs = codec.compress_chunked(x, 4, wl.eb.numpy())
    o = offs.cpu().tolist()
    for r, (b0, b1) in enumerate(oracle.chunk_rows(300, 4)):
        single, nb = codec.compress(x[b0:b1].contiguous(), wl.eb.numpy())
        n = int(nb.item())
        assert n == o[r + 1] - o[r]
        assert torch.equal(single[:n], out[o[r]:o[r + 1]])
        # and the plain decoder restores the slice from it
        xh = codec.decompress(out[o[r]:o[r + 1]].clone(), n, b1 - b0, *x.shape[1:])
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        xo, _ = oracle.decompress(out[o[r]:o[r + 1]].cpu().numpy(), b1 - b0, *x.shape[1:])
        assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))


def test_table_stats_sum_over_slices(codec):
    wl = workloads.make("fwd", batch=1200, tables=5)
    x = wl.x.cuda()
    codec.compress_chunked(x, 6, wl.eb.numpy())
    torch.cuda.synchronize()
    st = codec.table_stats(5)
    ref, roffs = oracle.compress_chunked(wl.x.numpy(), wl.eb.numpy(), 6)
    lits = [0] * 5
    for r in range(6):
        c = ref[int(roffs[r]):int(roffs[r + 1])]
        for t in range(5):
            rec = 144 + 272 * t
            lits[t] += int.from_bytes(bytes(c[rec + 4:rec + 8]), "little")
    assert [s["n_literal"] for s in st] == lits


def _decode_rc(codec, buf, in_bytes, offs, shape):
    xh = torch.empty(shape, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    rc = ebc.ebc_decompress_chunked(codec.handle, ctypes.c_void_p(buf.data_ptr()), in_bytes,
                                    ctypes.c_void_p(offs.data_ptr()), offs.numel() - 1, ctypes.c_void_p(xh.data_ptr()),
                                    *shape, None)
    assert rc == 0
    return codec.last_error()


def test_bad_boundaries_and_containers(codec):
    wl = workloads.make("tiny")
    x = wl.x.cuda()
    out, offs = codec.compress_chunked(x, 3, wl.eb.numpy())
    torch.cuda.synchronize()
    total = int(offs[-1].item())
    shape = tuple(x.shape)
    assert _decode_rc(codec, out, total, offs, shape) == 0
    bad = offs.clone()
    bad[1] += 8                                   # off a 16-byte boundary
    assert _decode_rc(codec, out, total, bad, shape) == ebc.EBC_ERR_CORRUPT
    bad = offs.clone()
    bad[3] = total + 16                           # past the input
    assert _decode_rc(codec, out, total, bad, shape) == ebc.EBC_ERR_CORRUPT
    bad = offs.clone()
    bad[1], bad[2] = offs[2], offs[1]             # decreasing
    assert _decode_rc(codec, out, total, bad, shape) == ebc.EBC_ERR_CORRUPT
    # the containers of 4 slices do not fit a 3-slice split of the same batch
    out4, offs4 = codec.compress_chunked(x, 4, wl.eb.numpy())
    torch.cuda.synchronize()
    rc = _decode_rc(codec, out4, int(offs4[-1].item()), offs4[:4].contiguous(), shape)
    assert rc in (ebc.EBC_ERR_INVALID_ARG, ebc.EBC_ERR_CORRUPT)
    # and the context still decodes a good buffer afterwards
    assert _decode_rc(codec, out, total, offs, shape) == 0


def test_windows_must_agree(codec):
    wl = workloads.make("tiny", batch=200)
    x = wl.x.cuda()
    codec.set_window(4)
    try:
        a, oa = codec.compress_chunked(x, 2, wl.eb.numpy())
    finally:
        codec.set_window(0)
    b, ob = codec.compress_chunked(x, 2, wl.eb.numpy())
    torch.cuda.synchronize()
    oa, ob = oa.cpu().tolist(), ob.cpu().tolist()
    # container 0 with a window, container 1 without
    mixed = torch.cat([a[oa[0]:oa[1]], b[ob[1]:ob[2]]])
    offs = torch.tensor([0, oa[1], oa[1] + ob[2] - ob[1]], dtype=torch.int64, device="cuda")
    assert _decode_rc(codec, mixed, int(offs[-1].item()), offs, tuple(x.shape)) == ebc.EBC_ERR_CORRUPT


def test_capacity(codec):
    wl = workloads.make("tiny")
    x = wl.x.cuda()
    full, offs = codec.compress_chunked(x, 3, wl.eb.numpy())
    torch.cuda.synchronize()
    need = int(offs[-1].item())
    small = torch.zeros(need - 16, dtype=torch.uint8, device="cuda")
    o2 = torch.zeros(4, dtype=torch.int64, device="cuda")
    rc = ebc.ebc_compress_chunked(codec.handle, ctypes.c_void_p(x.data_ptr()), *x.shape,
                                  np.ascontiguousarray(wl.eb.numpy()).ctypes.data_as(ctypes.c_void_p), 3,
                                  ctypes.c_void_p(small.data_ptr()), small.numel(), ctypes.c_void_p(o2.data_ptr()),
                                  None)
    assert rc == 0
    assert codec.last_error() == ebc.EBC_ERR_CAPACITY
    assert int(o2[-1].item()) == need


def test_receiving_side_columns_on_parallel_streams():
    # three senders (2, 3 and 4 tables; one with a window, one with the wide alphabet), each
    # container decoded into its columns of one [B, 9, D] output, each on its own stream
    B, D, T_out = 1500, 32, 9
    senders = [(2, 0, 128), (3, 16, 128), (4, 0, 512)]   # tables, window, radius
    out = torch.full((B, T_out, D), 7.0, dtype=torch.float32, device="cuda")
    ref = np.full((B, T_out, D), np.float32(7.0))
    keep = []
    col = 0
    for k, (Ts, win, rad) in enumerate(senders):
        x, eb = _dup_rows(B, Ts, D, seed=40 + k, pool=300)
        enc = ebc.Codec(0)
        enc.set_radius(rad)
        enc.set_window(win)
        buf, nb = enc.compress(torch.from_numpy(x).cuda(), eb)
        torch.cuda.synchronize()
        assert enc.last_error() == 0
        n = int(nb.item())
        enc.close()
        dec = ebc.Codec(0)
        dec.set_radius(rad)
        st = torch.cuda.Stream()
        dec.decompress_columns(buf, n, Ts, out, col, stream=st)
        keep.append((dec, st, buf))
        oracle.decompress_columns(buf[:n].cpu().numpy(), B, Ts, D, T_out, col, out=ref)
        col += Ts
    torch.cuda.synchronize()
    for dec, _, _ in keep:
        assert dec.last_error() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # columns outside the output are refused before any device work
    dec = keep[0][0]
    buf = keep[0][2]
    for Ts, t_off in ((2, 8), (2, -1)):
        rc = ebc.ebc_decompress_columns(dec.handle, ctypes.c_void_p(buf.data_ptr()), buf.numel(),
                                        ctypes.c_void_p(out.data_ptr()), B, Ts, D, T_out, t_off, None)
        assert rc == ebc.EBC_ERR_INVALID_ARG
    for dec, _, _ in keep:
        dec.close()
