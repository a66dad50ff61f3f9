"""Contexts created with an ebc_config, through the C ABI: each option gives
the container the oracle makes with the same option, byte for byte, and
ebc_get_stats reads the counts on a caller's stream."""
import ctypes

import numpy as np
import pytest
import torch

import error_bounded_lossy_gb300 as ebc
import oracle
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _roundtrip(codec, x_np, eb):
    x = torch.from_numpy(x_np).cuda()
    out, nb = codec.compress(x, eb)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    n = int(nb.item())
    buf = out[:n].cpu().numpy()
    xh = codec.decompress(out, n, *x_np.shape)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    return buf, xh.cpu().numpy()


@pytest.mark.parametrize("cfg,okw", [
    (None, {}),
    (dict(), {}),
    (dict(radius=512), {"radius": 512}),
    (dict(dedup=0), {"modes": "nodedup"}),
    (dict(window=32), {"window": 32}),
    (dict(radius=512, window=7, dedup=1), {"radius": 512, "window": 7}),
])
def test_config_options_match_the_oracle(cfg, okw):
    wl = workloads.make("fwd", batch=3000, tables=5)
    x_np, eb = wl.x.numpy(), wl.eb.numpy()
    codec = ebc.Codec(0, ebc.EbcConfig(**cfg) if cfg is not None else None)
    try:
        buf, xh = _roundtrip(codec, x_np, eb)
        kw = dict(okw)
        if kw.get("modes") == "nodedup":
            kw["modes"] = np.full(x_np.shape[1], oracle.MODE_HUFFMAN, np.uint8)
        ref, info = oracle.compress(x_np, eb, **kw)
        assert len(buf) == len(ref) and np.array_equal(buf, ref)
        xo, _ = oracle.decompress(ref, *x_np.shape)
        assert np.array_equal(xh.view(np.uint32), xo.view(np.uint32))
        # the counts, read on a caller's stream
        side = torch.cuda.Stream()
        rc, st = ebc.ebc_get_stats(codec.handle, ctypes.c_void_p(side.cuda_stream))
        assert rc == 0
        assert st.out_bytes == len(ref) and st.n_literal == info["n_literal"] and st.n_match == info["n_match"]
        if cfg and cfg.get("dedup") == 0:
            assert st.n_match == 0
    finally:
        codec.close()


def test_dedup_off_with_table_modes_on_top():
    """dedup = 0 makes every table a no-dedup table; raw codes set per table
    still apply."""
    wl = workloads.make("fwd", batch=2000, tables=4)
    x_np, eb = wl.x.numpy(), wl.eb.numpy()
    codec = ebc.Codec(0, ebc.EbcConfig(dedup=0))
    try:
        codec.set_table_modes(np.array([0, 2, 0, 2], np.uint8))
        buf, _ = _roundtrip(codec, x_np, eb)
        ref, _ = oracle.compress(x_np, eb, modes=np.array([1, 3, 1, 3], np.uint8))
        assert np.array_equal(buf, ref)
    finally:
        codec.close()
