"""ebc_decompress_noalloc: decoding without any device allocation.

Callers that cannot allocate while they decode (a process whose device memory
belongs to another allocator's pool, or a latency-bound loop where cudaMalloc
and cudaFree would synchronise the device) use this entry point; it keeps its
scratch in one static device array of the library.  These tests call it
through the C ABI and require the same reconstruction, bit for bit, as the
context-based ebc_decompress, on consecutive calls that share the array.

The file name makes pytest collect it after every other test file.
"""
import ctypes

import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(scope="module")
def codec():
    c = ebc.Codec(0)
    yield c
    c.close()


def _container(codec, name, **kw):
    """(container tensor, size, shape, reference xhat from ebc_decompress)."""
    wl = workloads.make(name, **kw)
    x = wl.x.to("cuda")
    out, nb = codec.compress(x, wl.eb.numpy())
    n = int(nb.item())
    ref = codec.decompress(out, n, *x.shape)
    torch.cuda.synchronize()
    codec.check()
    return out, n, tuple(x.shape), ref


def _noalloc(out, n, shape, stream=None):
    xhat = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    rc = ebc.ebc_decompress_noalloc(ctypes.c_void_p(out.data_ptr()), n, ctypes.c_void_p(xhat.data_ptr()),
                                    *shape, ctypes.c_void_p(stream.cuda_stream if stream else 0))
    return rc, xhat


def _same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_matches_ebc_decompress_on_consecutive_calls(codec):
    big = _container(codec, "fwd")
    small = _container(codec, "tiny")
    side = torch.cuda.Stream()
    # the second call finds the first call's tables in the shared array; the
    # third repeats the first on another stream
    for (out, n, shape, ref), stream in ((big, None), (small, None), (big, side)):
        rc, xhat = _noalloc(out, n, shape, stream)
        assert rc == ebc.EBC_OK, ebc.ebc_strerror(rc)
        assert _same_bits(xhat, ref)


def test_recovers_after_a_corrupt_container(codec):
    out, n, shape, ref = _container(codec, "tiny")
    bad = out.clone()
    bad[0] ^= 0xFF   # magic number
    rc, _ = _noalloc(bad, n, shape)
    assert rc in (ebc.EBC_ERR_CORRUPT, ebc.EBC_ERR_INVALID_ARG)
    rc, xhat = _noalloc(out, n, shape)
    assert rc == ebc.EBC_OK
    assert _same_bits(xhat, ref)


def test_rejects_a_shape_beyond_the_static_scratch():
    B, T, D = 1 << 20, 8, 4           # the reference-chain table alone needs 32 MiB
    src = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    xhat = torch.full((B, T, D), 7.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    rc = ebc.ebc_decompress_noalloc(ctypes.c_void_p(src.data_ptr()), src.numel(), ctypes.c_void_p(xhat.data_ptr()),
                                    B, T, D, None)
    assert rc == ebc.EBC_ERR_SCRATCH_LIMIT
    assert "static scratch" in ebc.ebc_strerror(rc)
    torch.cuda.synchronize()
    assert bool((xhat == 7.0).all())
