"""The C-ABI library builds, loads and exports every declared symbol; argument checks
return their status codes without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from sparse_attention_29_b300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(capi.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert capi.version().startswith("libdsa")


def test_status_strings(lib):
    for code in range(6):
        assert lib.dsa_status_string(code)
    assert lib.dsa_status_string(99) == b"unknown status"


def test_null_and_range_checks_fail_before_any_launch(lib):
    L = capi.CacheLayout(None, None, 0, 0, 0)
    INVALID, UNSUPPORTED = 1, 2
    # indexer: null pointers, zero sizes, unsupported head dim
    assert lib.dsa_indexer_scores(None, None, None, None, None, ctypes.byref(L), None,
                                  1, 1, 64, 128, 16, None, None) == INVALID
    p = 0x1000  # never dereferenced: the checks below fail first
    assert lib.dsa_indexer_scores(p, p, p, p, p, ctypes.byref(L), p, 0, 1, 64, 128, 16, p,
                                  None) == INVALID
    assert lib.dsa_indexer_scores(p, p, p, p, p, ctypes.byref(L), p, 1, 1, 64, 96, 16, p,
                                  None) == UNSUPPORTED
    # a layout with neither seq_start nor block table
    assert lib.dsa_indexer_scores(p, p, p, p, p, ctypes.byref(L), p, 1, 1, 64, 128, 16, p,
                                  None) == INVALID
    # misaligned key cache
    L2 = capi.CacheLayout(p, None, 0, 0, 100)
    assert lib.dsa_indexer_scores(p, p, p, p + 4, p, ctypes.byref(L2), p, 1, 1, 64, 128, 16,
                                  p, None) == INVALID
    # paged indexer needs page_size % 64 == 0
    L3 = capi.CacheLayout(None, p, 32, 4, 128)
    assert lib.dsa_indexer_scores(p, p, p, p, p, ctypes.byref(L3), p, 1, 1, 64, 128, 16, p,
                                  None) == INVALID
    # top-k: k out of range
    assert lib.dsa_topk(p, p, 4, 100, 0, p, None) == INVALID
    assert lib.dsa_topk(p, p, 4, 100, 9000, p, None) == UNSUPPORTED
    assert lib.dsa_topk(p, p, 4, 375041, 2048, p, None) == UNSUPPORTED  # longer than a cluster holds
    assert lib.dsa_topk_sparse_mla_decode(p, p, 375041, p, p, None, p, 4, 64, 512, 64, 2048,
                                          0.0625, p, p, p, 0, None) == UNSUPPORTED
    assert lib.dsa_topk(None, p, 4, 100, 64, p, None) == INVALID
    # sparse MLA: shapes outside the build
    assert lib.dsa_sparse_mla_decode(p, p, ctypes.byref(L2), p, 1, 128, 512, 64, 2048,
                                     ctypes.c_float(0.0625), p, None, None, 0,
                                     None) == UNSUPPORTED
    assert lib.dsa_sparse_mla_decode(p, p, ctypes.byref(L2), p, 1, 64, 500, 64, 2048,
                                     ctypes.c_float(0.0625), p, None, None, 0,
                                     None) == UNSUPPORTED
    assert lib.dsa_sparse_mla_decode(p, p, ctypes.byref(L2), p, 1, 64, 512, 64, 2048,
                                     ctypes.c_float(-1.0), p, None, None, 0, None) == INVALID
    assert lib.dsa_sparse_mla_decode(p + 8, p, ctypes.byref(L2), p, 1, 64, 512, 64, 2048,
                                     ctypes.c_float(0.0625), p, None, None, 0,
                                     None) == INVALID
    assert lib.dsa_sparse_mla_shared(None, None, 0, ctypes.byref(L2), p, 1, 1, 64, 512, 64,
                                     2048, ctypes.c_float(0.0625), None, None, None, 0,
                                     None) == INVALID


def test_workspace_query_without_gpu(lib):
    assert lib.dsa_workspace_bytes(0, 1, 1, 64, 512, 2048, 1) == 0
    assert lib.dsa_workspace_bytes(1, 1, 1, 64, 512, 2048, 1) == 0
    assert lib.dsa_workspace_bytes(2, 0, 1, 64, 512, 2048, 1) == ctypes.c_size_t(-1).value


def test_layout_keeps_its_tensors_alive():
    """The layout structure holds raw addresses, so it must keep its tensors referenced."""
    import gc
    import weakref
    import torch
    from sparse_attention_29_b300 import capi
    t = torch.arange(4, dtype=torch.int32)
    ref = weakref.ref(t)
    layout = capi.make_layout(10, seq_start=t)
    del t
    gc.collect()
    assert ref() is not None and layout.seq_start == ref().data_ptr()


def test_fused_indexer_topk_checks_fail_before_any_launch(lib):
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 4
    p = 0x1000
    L2 = capi.CacheLayout(p, None, 0, 0, 100)
    need = lib.dsa_indexer_topk_workspace_bytes(1, 16, 100)
    assert need == 16 * 128 * 8 + 16 * 32
    assert lib.dsa_indexer_topk_workspace_bytes(0, 16, 100) == ctypes.c_size_t(-1).value
    args = (p, p, p, p, p, ctypes.byref(L2), p, 1, 16, 64, 128, 100, 32)
    assert lib.dsa_indexer_topk(*args, None, p, need, None) == INVALID        # no output
    assert lib.dsa_indexer_topk(*args, p, p, need - 16, None) == WORKSPACE    # too small
    assert lib.dsa_indexer_topk(*args, p, p + 8, need, None) == INVALID       # misaligned
    assert lib.dsa_indexer_topk(p, p, p, p, p, ctypes.byref(L2), p, 1, 16, 64, 128, 100, 9000,
                                p, p, need, None) == UNSUPPORTED              # k too large
    assert lib.dsa_indexer_topk(p, p, p, p, p, ctypes.byref(L2), p, 1, 16, 16, 128, 100, 32,
                                p, p, need, None) == UNSUPPORTED              # 16 heads: > 4 rows a tile


def test_hisparse_checks_fail_before_any_launch(lib):
    INVALID, UNSUPPORTED = 1, 2
    p = 0x1000
    U32 = ctypes.c_uint32
    # null arguments, step 0, a working set smaller than the selection, sizes past the build
    assert lib.dsa_hisparse_fetch(None, 1, 8, U32(1), p, p, 576, p, 100, p, p, 16, p, None,
                                  None) == INVALID
    assert lib.dsa_hisparse_fetch(p, 1, 8, U32(0), p, p, 576, p, 100, p, p, 16, p, None,
                                  None) == INVALID
    assert lib.dsa_hisparse_fetch(p, 1, 32, U32(1), p, p, 576, p, 100, p, p, 16, p, None,
                                  None) == INVALID
    assert lib.dsa_hisparse_fetch(p, 1, 8, U32(1), p, p, 570, p, 100, p, p, 16, p, None,
                                  None) == INVALID                         # D % 8 != 0
    assert lib.dsa_hisparse_fetch(p, 1, 9000, U32(1), p, p, 576, p, 100000, p, p, 9000, p,
                                  None, None) == UNSUPPORTED
    assert lib.dsa_hisparse_init(p, 1, 100, p, p, 20000, None) == UNSUPPORTED
    assert lib.dsa_hisparse_init(None, 1, 100, p, p, 16, None) == INVALID
    # the wait probe: a result pointer is required and must be 8-byte aligned
    assert lib.dsa_wait_probe(None, None) == INVALID
    assert lib.dsa_wait_probe(ctypes.c_void_p(4100), None) == INVALID
