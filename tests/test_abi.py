"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
entry point that include/ebc.h declares; host-only calls behave as documented."""
import ctypes
import os
import re

import pytest

import error_bounded_lossy_gb300 as ebc
import oracle
from error_bounded_lossy_gb300 import build as ebc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ebc_build.build()
    return ebc.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ebc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ebc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ebc_compress", "ebc_decompress", "ebc_set_error_bounds"):
        assert required in names
    assert set(names) == set(ebc.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {ebc.library_path()}").read()
    exported = set(re.findall(r"\bT (ebc_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported


def test_host_only_calls(lib):
    assert ebc.ebc_version() == 1
    for code in range(8):
        assert ebc.ebc_strerror(code)
    assert ebc.ebc_strerror(99) == "unknown error"
    # unsupported shapes
    assert ebc.ebc_compress_bound(10, 2, 24) == 0
    assert ebc.ebc_compress_bound(10, 2000, 16) == 0
    assert ebc.ebc_compress_bound(1 << 24, 1, 16) == 0
    # the worst-case bound agrees with the oracle's and covers real containers
    for shape in [(0, 3, 16), (1, 1, 4), (512, 4, 16), (8192, 26, 128), (65536, 26, 256), (33, 2, 512)]:
        assert ebc.ebc_compress_bound(*shape) == oracle.compress_bound(*shape)


def test_create_without_device_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.ebc_create(ctypes.byref(h), None, 0) == ebc.EBC_ERR_NO_DEVICE
    assert not h.value
    assert lib.ebc_last_device_error(None) == ebc.EBC_ERR_INVALID_ARG


def test_bounds_of_the_wide_alphabet_and_of_chunked_buffers(lib):
    # the wide alphabet's bound agrees with the oracle's (1040-byte table records)
    for shape in [(0, 3, 16), (1, 1, 4), (512, 4, 16), (8192, 26, 128), (33, 2, 512)]:
        assert ebc.ebc_compress_bound_radius(*shape, 512) == oracle.compress_bound(*shape, radius=512)
        assert ebc.ebc_compress_bound_radius(*shape, 128) == ebc.ebc_compress_bound(*shape)
    assert ebc.ebc_compress_bound_radius(512, 4, 16, 256) == 0
    # a chunked buffer's bound is the sum of its slices' bounds (numpy array_split slices)
    for B, T, D, n in [(8192, 26, 128, 8), (1001, 3, 8, 7), (3, 2, 16, 5), (0, 4, 16, 4), (65537, 1, 4, 2)]:
        for radius in (128, 512):
            want = sum(oracle.compress_bound(b1 - b0, T, D, radius) for b0, b1 in oracle.chunk_rows(B, n))
            assert ebc.ebc_compress_chunked_bound(B, T, D, n, radius) == want
    assert ebc.ebc_compress_chunked_bound(100, 2, 16, 0, 128) == 0
    assert ebc.ebc_compress_chunked_bound(100, 2, 16, ebc.EBC_MAX_CHUNKS + 1, 128) == 0
    assert ebc.ebc_compress_chunked_bound(100, 2, 24, 2, 128) == 0
    assert ebc.ebc_compress_chunked_bound(100, 2, 16, 2, 300) == 0


def test_chunked_and_radius_calls_reject_bad_arguments_before_any_device_work(lib):
    # a null context is refused by every new entry point
    assert ebc.ebc_set_radius(None, 512) == ebc.EBC_ERR_INVALID_ARG
    assert ebc.ebc_compress_chunked(None, None, 8, 2, 16, None, 2, None, 0, None, None) == ebc.EBC_ERR_INVALID_ARG
    assert ebc.ebc_compress_chunked_bf16(None, None, 8, 2, 16, None, 2, None, 0, None, None) == \
        ebc.EBC_ERR_INVALID_ARG
    assert ebc.ebc_decompress_chunked(None, None, 0, None, 2, None, 8, 2, 16, None) == ebc.EBC_ERR_INVALID_ARG


def test_config_path_through_ctypes(lib):
    """ebc_config: NULL and EBC_CONFIG_DEFAULT agree; the radius changes the
    bound as the oracle's does; values the container format does not allow are
    refused before any device is touched."""
    default = ebc.EbcConfig()
    assert (default.radius, default.chunk_vectors, default.max_code_len, default.dedup, default.window) == \
        (128, 0, 24, 1, 0)
    for shape in [(0, 3, 16), (512, 4, 16), (8192, 26, 128), (33, 2, 512)]:
        assert ebc.ebc_compress_bound(*shape, default) == ebc.ebc_compress_bound(*shape) == oracle.compress_bound(*shape)
        assert ebc.ebc_compress_bound(*shape, ebc.EbcConfig(radius=512)) == oracle.compress_bound(*shape, radius=512)
        assert ebc.ebc_compress_bound(*shape, ebc.EbcConfig(radius=0)) == oracle.compress_bound(*shape)
        # dedup and window do not change the worst case
        assert ebc.ebc_compress_bound(*shape, ebc.EbcConfig(dedup=0, window=64)) == oracle.compress_bound(*shape)
    bad = [ebc.EbcConfig(radius=256), ebc.EbcConfig(chunk_vectors=4), ebc.EbcConfig(max_code_len=16),
           ebc.EbcConfig(dedup=2), ebc.EbcConfig(window=256), ebc.EbcConfig(window=-1)]
    for cfg in bad:
        assert ebc.ebc_compress_bound(512, 4, 16, cfg) == 0
        h = ctypes.c_void_p()
        assert lib.ebc_create(ctypes.byref(h), ctypes.byref(cfg), 0) == ebc.EBC_ERR_INVALID_ARG
        assert not h.value
    # a good config reaches the device check (no GPU here: NO_DEVICE; with one: a context)
    import torch
    if not torch.cuda.is_available():
        h = ctypes.c_void_p()
        assert lib.ebc_create(ctypes.byref(h), ctypes.byref(ebc.EbcConfig(radius=512)), 0) == ebc.EBC_ERR_NO_DEVICE
    # null arguments
    assert lib.ebc_get_stats(None, None, None) == ebc.EBC_ERR_INVALID_ARG
