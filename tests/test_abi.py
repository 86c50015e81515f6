"""The C-ABI library: builds, loads without a GPU, exports every declared
symbol, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_decode_gb300 import build as b
    path = b.build()
    import compressed_sparse_attention_decode_gb300 as csa
    return csa.load(path)


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared()
    for n in ("csa2_cache_write", "csa2_indexer_topk", "csa2_reindex", "csa2_sparse_attn", "csa2_quantize_fp4",
              "csa2_workspace_size", "csa2_status_string", "csa2_abi_version", "csa2_launch_count"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import compressed_sparse_attention_decode_gb300 as csa
    out = subprocess.run(["nm", "-D", "--defined-only", csa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s+(\S+)", out))
    for n in declared():
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(csa.EXPORTS) == set(declared())


def test_host_side_validation_needs_no_gpu(lib):
    import compressed_sparse_attention_decode_gb300 as csa
    assert lib.csa2_abi_version() == 200
    assert lib.csa2_status_string(1) == b"invalid argument"
    # NULL cache / bad sizes are refused before any CUDA call
    assert lib.csa2_cache_write(None, None, 0, 0, None, None, None, None) == csa.ERR_INVALID_ARG
    c = csa._CacheStruct(16, 16, 16, 16, 1, 8, 512, 128, 2)
    assert lib.csa2_cache_write(ctypes.byref(c), ctypes.c_void_p(16), 1, 2, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), None, None) == csa.ERR_INVALID_ARG     # odd pos0
    assert lib.csa2_cache_write(ctypes.byref(c), ctypes.c_void_p(16), 0, 18, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), None, None) == csa.ERR_INVALID_ARG     # beyond capacity
    bad = csa._CacheStruct(16, 16, 16, 16, 1, 8, 256, 128, 2)
    assert lib.csa2_sparse_attn(ctypes.byref(bad), None, 1, 1, None, None, 0, None, 0, 0, 1.0, None, None, None,
                                0, None) == csa.ERR_UNSUPPORTED
    p = ctypes.c_void_p(256)
    assert lib.csa2_sparse_attn(ctypes.byref(c), p, 1, 0, p, p, 4, p, 0, 128, 1.0, p, None, None, 0,
                                None) == csa.ERR_INVALID_ARG                                  # zero heads
    assert lib.csa2_indexer_topk(ctypes.byref(c), p, p, p, 1, p, 8, 4096, p, 0, 8, None, p, 1 << 30,
                                 None) == csa.ERR_INVALID_ARG                                 # k too large
    assert lib.csa2_indexer_topk(ctypes.byref(c), p, p, p, 1, p, 8, 64, p, 0, 8, None, p, 0,
                                 None) == csa.ERR_WORKSPACE                                   # no workspace
    assert lib.csa2_reindex(7, ctypes.byref(c), p, p, p, 1, 8, p, 8, p, 4, p, None, 0, None) == csa.ERR_INVALID_ARG
    # Reindex from fp32 queries: NULL or misaligned queries, bad pool sizes, missing workspace
    assert lib.csa2_reindex_f32(ctypes.byref(c), None, p, 1, 8, p, 8, 4, p, p, 1 << 30, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_reindex_f32(ctypes.byref(c), ctypes.c_void_p(260), p, 1, 8, p, 8, 4, p, p, 1 << 30,
                                None) == csa.ERR_INVALID_ARG                                  # iq not 16-aligned
    assert lib.csa2_reindex_f32(ctypes.byref(c), p, p, 1, 8, p, 0, 4, p, p, 1 << 30, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_reindex_f32(ctypes.byref(c), p, p, 1, 8, p, 8, 4, p, None, 0, None) == csa.ERR_WORKSPACE
    assert lib.csa2_quantize_fp4(p, 4, 24, p, p, None) == csa.ERR_INVALID_ARG                  # d not /16
    assert lib.csa2_workspace_size(csa.OP_INDEXER_TOPK, 2, 1, 8, 512, 1000) > 0
    assert lib.csa2_launch_count() >= 0
    # failure detection: NULL, short or misaligned workspaces and a zero poll limit are refused
    assert lib.csa2_poll_error(None, 16, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_poll_error(p, 8, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_poll_error(ctypes.c_void_p(264), 64, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_selftest_wait_timeout(0, p, 64, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_selftest_wait_timeout(16, None, 64, None) == csa.ERR_INVALID_ARG
    assert lib.csa2_status_string(csa.ERR_TIMEOUT) == b"a kernel gave up on a bounded wait"


def test_binding_fails_loudly_without_the_library(tmp_path):
    import compressed_sparse_attention_decode_gb300 as csa
    with pytest.raises(RuntimeError, match="not built"):
        csa.load(str(tmp_path / "missing.so"))
