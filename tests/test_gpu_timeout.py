"""Failure detection on the GPU without a fault: the bounded wait of the
quantize kernel's first input tile is given zero polls, so every block gives up
at once, records EBC_ERR_DEVICE_TIMEOUT, waits (with the full limit) for the
tile copies it had issued, and stops; the later kernels of the call write
nothing to the output.  The host reads the status, and the same context then
compresses byte-exact again.  Nothing hangs: the only waits that run out are
the ones set to zero."""
import numpy as np
import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import oracle
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("fwd", {"batch": 4096})])
def test_first_wait_runs_out_and_the_context_recovers(name, kw):
    wl = workloads.make(name, **kw)
    x, eb = wl.x.cuda(), wl.eb.numpy()
    ref, _ = oracle.compress(wl.x.numpy(), eb)
    codec = ebc.Codec(0)
    try:
        assert ebc.ebc_set_first_wait_polls(codec.handle, 0) == 0
        sentinel = 0x5A
        out = torch.full((codec.compress_bound(*wl.shape),), sentinel, dtype=torch.uint8, device="cuda")
        nb = torch.zeros(1, dtype=torch.int64, device="cuda")
        codec.compress_into(x, eb, out, nb)
        torch.cuda.synchronize()
        assert codec.last_error() == ebc.EBC_ERR_DEVICE_TIMEOUT
        # a given-up call writes nothing past the container's fixed-size header
        assert (out[144:].cpu().numpy() == sentinel).all()
        assert codec.last_error() == 0          # the status was read once and cleared
        # the full limit again: the same context compresses as before
        assert ebc.ebc_set_first_wait_polls(codec.handle, -1) == 0
        out2, nb2 = codec.compress(x, eb)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        n = int(nb2.item())
        assert n == len(ref) and np.array_equal(out2[:n].cpu().numpy(), ref)
        xh = codec.decompress(out2, n, *wl.shape)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        xo, _ = oracle.decompress(ref, *wl.shape)
        assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
    finally:
        codec.close()


def test_wait_limit_argument_checks():
    codec = ebc.Codec(0)
    try:
        assert ebc.ebc_set_first_wait_polls(codec.handle, (1 << 22) + 1) == ebc.EBC_ERR_INVALID_ARG
        assert ebc.ebc_set_first_wait_polls(None, 0) == ebc.EBC_ERR_INVALID_ARG
        assert ebc.ebc_set_first_wait_polls(codec.handle, 1 << 22) == 0
    finally:
        codec.close()
