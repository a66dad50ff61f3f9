"""Native bf16 input on the GPU (ebc_compress_bf16), against the oracle.

A bf16 batch is coded as its exact fp32 values, so its container must be
byte-identical to the oracle's container of the fp32-converted batch, and the
reconstruction 0 ulp from the oracle's ("Accelerating Communication in Deep
Learning Recommendation Model Training with Dual-Level Adaptive Lossy
Compression", §III-D; the mixed-precision training of §IV)."""
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


def _check(codec, xb, eb):
    x32 = xb.float().numpy()
    out, nb = codec.compress(xb.cuda(), eb)
    torch.cuda.synchronize()
    assert codec.last_error() == 0
    n = int(nb.item())
    buf = out[:n].cpu().numpy()
    ref, info = oracle.compress(x32, eb)
    assert len(buf) == len(ref) and np.array_equal(buf, ref)
    xh = codec.decompress(out, n, *x32.shape)
    torch.cuda.synchronize()
    xo, _ = oracle.decompress(ref, *x32.shape)
    assert np.array_equal(xh.cpu().numpy().view(np.uint32), xo.view(np.uint32))
    return info


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("fwd", {}), ("bwd", {"batch": 4096}),
                                     ("large", {"batch": 2048, "variant": "bf16"})])
def test_bf16_workloads(codec, name, kw):
    wl = workloads.make(name, **kw)
    _check(codec, wl.x.to(torch.bfloat16), wl.eb.numpy())


@pytest.mark.parametrize("D", [8, 16, 64, 256, 512])
@pytest.mark.parametrize("B", [1, 33, 1000])
def test_bf16_shapes_with_outliers(codec, B, D):
    rng = np.random.default_rng(B * 7 + D)
    T = 3
    x = rng.normal(0, 0.05, size=(B, T, D)).astype(np.float32)
    x[rng.random(size=x.shape) < 0.01] *= 1e4      # outliers: raw bits through the bf16 path
    if B > 4:
        x[B // 2:] = x[: B - B // 2]                  # duplicates, compared on the raw outlier bits
    eb = np.full(T, 1e-3, np.float32)
    _check(codec, torch.from_numpy(x).to(torch.bfloat16), eb)


def test_bf16_needs_d8(codec):
    x = torch.zeros((16, 2, 4), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ebc.EbcError) as e:
        codec.compress(x, np.full(2, 1e-3, np.float32))
    assert e.value.code == ebc.EBC_ERR_INVALID_ARG
