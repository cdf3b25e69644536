"""The C-ABI library loads, exports every symbol include/csa2.h declares, and
rejects bad arguments on the host before touching a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_layer_gb300 import build, csa2
    build.build()
    return csa2.load()


def _declared():
    with open(HEADER) as f:
        src = f.read()
    return sorted(set(re.findall(r"CSA2_API\s+[\w\s\*]+?\b(csa2_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["csa2_compress", "csa2_quant_mxfp4", "csa2_quant_fp8", "csa2_index_scores", "csa2_topk",
              "csa2_sparse_attn", "csa2_layer"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from compressed_sparse_attention_layer_gb300 import csa2
    for n in _declared():
        assert hasattr(lib, n), n
        assert n in csa2.EXPORTS, n


def test_status_strings(lib):
    for s in range(-8, 1):
        assert lib.csa2_status_string(s)
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(-99) == b"unknown status"


def test_host_validation_without_gpu(lib):
    from compressed_sparse_attention_layer_gb300 import csa2
    # shape errors are caught before any launch
    assert lib.csa2_compress(None, None, None, 0, 10, None, None) == -2
    assert lib.csa2_compress(None, None, None, 2, 1, None, None) == 0          # nothing to compress
    assert lib.csa2_compress(None, None, None, 2, 8, None, None) == -1
    assert lib.csa2_quant_fp8(None, 4, 100, None, None, None, 64, None, None) == -2
    assert lib.csa2_quant_fp8(None, 0, 128, None, None, None, 64, None, None) == 0
    assert lib.csa2_quant_mxfp4(None, 4, None, None, None, 64, None, None) == -1
    assert lib.csa2_quant_mxfp4(ctypes.c_void_p(16), 100, None, ctypes.c_void_p(16), ctypes.c_void_p(16), 64,
                                None, None) == -4                                # rows beyond the cache
    assert lib.csa2_quant_mxfp4(ctypes.c_void_p(8), 4, None, ctypes.c_void_p(16), ctypes.c_void_p(16), 64,
                                None, None) == -8                                # misaligned input
    assert lib.csa2_quant_fp4_e4m3(None, 4, None, None, None, 64, None, None) == -1
    assert lib.csa2_quant_fp4_e4m3(ctypes.c_void_p(8), 4, None, ctypes.c_void_p(16), ctypes.c_void_p(16), 64,
                                   None, None) == -8
    assert lib.csa2_topk(None, 10, None, 1, None, 0, None, None) == -2
    assert lib.csa2_topk(None, 10, None, 1, None, 5000, None, None) == -2
    assert lib.csa2_topk_blocks(None, 10, None, 1, 4096, None, None, None) == -2
    cache = csa2.Cache()
    batch = csa2.Batch()
    io = csa2.LayerIO()
    assert lib.csa2_layer(7, ctypes.byref(cache), ctypes.byref(batch), ctypes.byref(io), None, 0, None) == -3
    assert lib.csa2_layer(0, ctypes.byref(cache), ctypes.byref(batch), ctypes.byref(io), None, 0, None) == -1
    cache = csa2.Cache(16, 16, 16, 16, 100, 16, 4, 0, None)  # num_slots not a multiple of 64
    assert lib.csa2_index_scores(ctypes.byref(cache), ctypes.byref(batch), 16, 16, 16, None, None, 8, None) == -2
    cache = csa2.Cache(16, 16, 16, 16, 256, 16, 4, 0, None)
    batch = csa2.Batch(1, 1, 1, 0, 1000, 16, 16)             # more entries than 4 pages hold
    assert lib.csa2_index_scores(ctypes.byref(cache), ctypes.byref(batch), 16, 16, 16, None, None, 1000, None) == -4
    cache = csa2.Cache(16, 16, 16, 16, 256, 16, 4, 7, None)  # unknown main-KV format
    batch = csa2.Batch(1, 1, 1, 0, 100, 16, 16)
    assert lib.csa2_index_scores(ctypes.byref(cache), ctypes.byref(batch), 16, 16, 16, None, None, 104, None) == -3


def test_workspace_sizes(lib):
    from compressed_sparse_attention_layer_gb300 import csa2
    b = csa2.Batch(8, 1, 1, 0, 1 << 20, None, None)
    full = lib.csa2_layer_workspace_size(0, ctypes.byref(b))
    reindex = lib.csa2_layer_workspace_size(1, ctypes.byref(b))
    reuse = lib.csa2_layer_workspace_size(2, ctypes.byref(b))
    assert full >= 8 * (1 << 20) * 4 + 8 * (1 << 17) * 4 + 8 * 16384 * 4
    assert full > reindex >= 8 * 16384 * 4 and reuse < reindex
    assert lib.csa2_layer_workspace_size(5, ctypes.byref(b)) == 0
