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


def test_binding_constants_match_the_header():
    """Every integer constant the header defines and the binding mirrors under
    the same name (without the CSA2_ prefix) has the same value there."""
    from compressed_sparse_attention_layer_gb300 import csa2
    with open(HEADER) as f:
        src = f.read()
    defs = {m.group(1): int(m.group(2)) for m in
            re.finditer(r"#define\s+CSA2_(\w+)\s+\(?\s*(-?\d+)u?\s*\)?", src)}
    mirrored = [n for n in defs if hasattr(csa2, n)]
    for n in mirrored:
        assert getattr(csa2, n) == defs[n], (n, getattr(csa2, n), defs[n])
    for n in ("ATTN_DEDUP_WINDOW", "ATTN_EARLY_INPUTS", "ATTN_EARLY_ALL", "ATTN_SCHEDULE_CHUNKS",
              "ATTN_SCHEDULE_ROWS", "LAYER_SCORES_BF16", "LAYER_INDEX_E4M3_QUERY"):
        assert n in mirrored, n


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
    big = 1 << 31                                   # more rows than one launch grid covers
    assert lib.csa2_quant_mxfp4(ctypes.c_void_p(16), big, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                ctypes.c_void_p(16), 64, None, None) == -2
    assert lib.csa2_quant_fp4_e4m3(ctypes.c_void_p(16), big, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), 64, None, None) == -2
    assert lib.csa2_quant_fp8(ctypes.c_void_p(16), big, 128, ctypes.c_void_p(16), ctypes.c_void_p(16),
                              ctypes.c_void_p(16), 64, None, None) == -2
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


def test_layer_option_flags_validated_on_the_host(lib):
    """Unknown csa2_layer_io.flags or csa2_swa.flags bits are refused before any
    launch (fake aligned device pointers: nothing is dereferenced)."""
    from compressed_sparse_attention_layer_gb300 import csa2
    P = ctypes.c_void_p(1 << 12)
    cache = csa2.Cache(P, P, P, P, 1 << 12, P, 64, 0, None)
    batch = csa2.Batch(1, 1, 1, 0, 1000, P, P)
    def io(layer_flags=0, swa_flags=0, new_rows=None):
        s = csa2.Swa(P, P, 128, swa_flags, None, new_rows, None, 0.0, 0)
        return csa2.LayerIO(P, P, P, s, 1.0, layer_flags, P, P, P, P, P, None, None)
    both = csa2.ATTN_SCHEDULE_CHUNKS | csa2.ATTN_SCHEDULE_ROWS
    for bad in (io(layer_flags=4), io(layer_flags=1 << 30), io(swa_flags=32), io(swa_flags=both)):
        assert lib.csa2_layer(csa2.MODES["full"], ctypes.byref(cache), ctypes.byref(batch), ctypes.byref(bad),
                              P, 1 << 30, None) == -3
    # a negative RoPE base is a shape error
    s = csa2.Swa(P, P, 128, 0, None, None, None, -1.0, 0)
    neg = csa2.LayerIO(P, P, P, s, 1.0, 0, P, P, P, P, P, None, None)
    assert lib.csa2_layer(csa2.MODES["reuse"], ctypes.byref(cache), ctypes.byref(batch), ctypes.byref(neg),
                          P, 1 << 30, None) == -2


def test_attention_schedule_choice(lib):
    """csa2_sparse_attn_schedule: fewer than 40 query rows -> one cluster per
    key chunk and a merge; 40 or more -> persistent clusters over whole rows;
    the flags force either; refusals as the attention call itself (host only,
    fake pointers)."""
    from compressed_sparse_attention_layer_gb300 import csa2
    P = ctypes.c_void_p(1 << 12)
    def sched(batch, nq, flags=0, new_rows=None):
        b = csa2.Batch(batch, nq, 1, 0, 1000, P, P)
        s = csa2.Swa(P, P, 256, flags, None, new_rows, None, 0.0, 0)
        return lib.csa2_sparse_attn_schedule(ctypes.byref(b), ctypes.byref(s))
    C, R = csa2.ATTN_SCHEDULE_CHUNKS, csa2.ATTN_SCHEDULE_ROWS
    assert sched(8, 1) == C and sched(39, 1) == C and sched(8, 1, new_rows=P) == C and sched(8, 4) == C
    assert sched(40, 1) == R and sched(10, 4) == R and sched(1, 8192) == R and sched(64, 1, new_rows=P) == R
    assert sched(64, 1, flags=C) == C and sched(1, 1, flags=R) == R and sched(1, 1, flags=R, new_rows=P) == R
    assert sched(8, 1, flags=C | R) == -3 and sched(8, 4, new_rows=P) == -3
    assert sched(0, 1) == -2
    assert lib.csa2_sparse_attn_schedule(None, None) == -1


def test_workspace_sizes(lib):
    from compressed_sparse_attention_layer_gb300 import csa2
    b = csa2.Batch(8, 1, 1, 0, 1 << 20, None, None)
    full = lib.csa2_layer_workspace_size(0, ctypes.byref(b))
    reindex = lib.csa2_layer_workspace_size(1, ctypes.byref(b))
    reuse = lib.csa2_layer_workspace_size(2, ctypes.byref(b))
    assert full >= 8 * (1 << 20) * 4 + 8 * (1 << 17) * 4
    # Reindex adds its rescored pool (16,384 keys and 32 group minima per row, 4 bytes each)
    # to the attention's scratch, which is all a Reuse layer needs
    assert full > reindex > reuse > 0
    assert reindex - reuse >= 8 * (16384 + 32) * 4
    assert lib.csa2_layer_workspace_size(5, ctypes.byref(b)) == 0


def test_append_entries_validated_on_the_host(lib):
    """csa2_append_entries refuses a missing cache or input, a bad group size,
    an unmapped overrun of the cache and a misaligned key array before any
    launch, and does nothing for fewer tokens than one group (fake pointers,
    never dereferenced)."""
    from compressed_sparse_attention_layer_gb300 import csa2
    P = ctypes.c_void_p(1 << 12)
    cache = ctypes.byref(csa2.Cache(P, P, P, P, 64, P, 1, 0, None))
    f = lib.csa2_append_entries
    assert f(None, P, P, P, 1, 8, P, None, None, None) == -1               # no cache
    assert f(cache, P, P, P, 0, 8, P, None, None, None) == -2              # m = 0
    assert f(cache, P, P, P, 17, 40, P, None, None, None) == -2            # m > 16
    assert f(cache, P, P, P, 4, 3, P, None, None, None) == 0               # no whole group: nothing to do
    assert f(cache, None, P, P, 1, 8, P, None, None, None) == -1           # no C
    assert f(cache, P, P, P, 1, 8, None, None, None, None) == -1           # no indexer keys
    assert f(cache, P, P, P, 1, 65, P, None, None, None) == -4             # 65 entries, 64 slots, no slot map
    assert f(cache, P, P, P, 1, 8, ctypes.c_void_p((1 << 12) + 4), None, None, None) == -8


def test_norm_rope_validated_on_the_host(lib):
    """csa2_norm_rope refuses bad shapes, missing or doubled outputs and
    misaligned pointers before any launch (fake pointers, never dereferenced)."""
    P, Q = ctypes.c_void_p(1 << 12), ctypes.c_void_p((1 << 12) + 8)
    f = lib.csa2_norm_rope
    assert f(P, 0, 64, None, 1e-6, None, 1e4, P, None, None) == 0               # nothing to do
    assert f(P, -1, 64, None, 1e-6, P, 1e4, P, None, None) == -2
    assert f(P, 4, 0, None, 1e-6, P, 1e4, P, None, None) == -2
    assert f(P, 1 << 30, 1 << 4, None, 1e-6, P, 1e4, P, None, None) == -2       # 2^34 vectors
    assert f(P, (1 << 30) - 1, 1 << 4, None, 1e-6, None, 0.0, None, None, None) == -1   # 2^34 - 16: in range
    assert f(P, 1 << 62, 1 << 30, None, 1e-6, P, 1e4, P, None, None) == -2      # the product would overflow
    assert f(P, 4, 64, None, -1e-6, P, 1e4, P, None, None) == -2
    assert f(P, 4, 64, None, float("nan"), P, 1e4, P, None, None) == -2
    assert f(P, 4, 64, None, 1e-6, P, -1.0, P, None, None) == -2
    assert f(P, 4, 64, None, 1e-6, P, float("inf"), P, None, None) == -2
    assert f(None, 4, 64, None, 1e-6, P, 1e4, P, None, None) == -1
    assert f(P, 4, 64, None, 1e-6, None, 1e4, P, None, None) == -1              # RoPE needs positions
    assert f(P, 4, 64, None, 1e-6, P, 1e4, None, None, None) == -1              # no output
    assert f(P, 4, 64, None, 1e-6, P, 1e4, P, P, None) == -1                    # two outputs
    assert f(Q, 4, 64, None, 1e-6, P, 1e4, P, None, None) == -8                # x not 16-byte aligned
    assert f(P, 4, 64, Q, 1e-6, P, 1e4, P, None, None) == -8                    # gamma
    assert f(P, 4, 64, None, 1e-6, P, 1e4, Q, None, None) == -8                 # fp32 output
    assert f(P, 4, 64, None, 1e-6, P, 1e4, None, ctypes.c_void_p((1 << 12) + 4), None) == -8
