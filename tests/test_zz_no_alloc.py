"""csa2_layer_noalloc: the layer call for callers that cannot allocate.

A caller that cannot hand the library a workspace buffer (a plugin whose host
program owns all device memory, a serving loop that allocates nothing after
start-up) uses this entry point; its scratch is a static device array of
CSA2_NOALLOC_SCRATCH_BYTES inside the library.  These checks compare it with
csa2_layer given a caller workspace, on the same inputs, for two passes with
an unrelated workload run through the array in between (the array keeps the
previous call's contents, so the second pass starts from unrelated data), and
check that work too large for the array is refused before anything runs.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from compressed_sparse_attention_layer_gb300 import csa2
from compressed_sparse_attention_layer_gb300 import workloads as W
from compressed_sparse_attention_layer_gb300.device import DeviceWorkload
from tests.reference import attn_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    from compressed_sparse_attention_layer_gb300 import build
    build.build()
    csa2.load()


def _run(dw, use_noalloc):
    dw.idx.fill_(-1)
    dw.pool.fill_(-1)
    dw.pool_len.zero_()
    out = {}
    for l in dw.layers:
        dw.o[l].fill_(np.nan)
        dw.lse[l].fill_(np.nan)
        mode = csa2.MODES[dw.wl.layers[l]]
        if use_noalloc:
            csa2.csa2_layer_noalloc(mode, dw.cstruct, dw.batch, dw.io(l))
        else:
            dw.run_layer(l)
        torch.cuda.synchronize()
        out[l] = (dw.idx.cpu().numpy().copy(), dw.pool_len.cpu().numpy().copy(),
                  dw.o[l].cpu().numpy().copy(), dw.lse[l].cpu().numpy().copy())
    return out


def _same(got, want, tag):
    for l in want:
        assert np.array_equal(got[l][0], want[l][0]), (tag, l, "indices")
        assert np.array_equal(got[l][1], want[l][1]), (tag, l, "pool sizes")
        for r in range(got[l][2].shape[0]):
            ok, info = attn_close(got[l][2][r], got[l][3][r], want[l][2][r], want[l][3][r])
            assert ok, (tag, l, r, info)
        # the kernels are deterministic: the scratch's earlier contents change no bit
        assert np.array_equal(got[l][2].view(np.int32), want[l][2].view(np.int32)), (tag, l, "o bits")
        assert np.array_equal(got[l][3].view(np.int32), want[l][3].view(np.int32)), (tag, l, "lse bits")


def test_noalloc_layer_matches_layer_twice():
    wl = W.Workload("noalloc", 4242, 3, [4096, 2500, 20000], 1,
                    ["full", "reuse", "reindex", "reuse"], planted_blocks=4)
    dw = DeviceWorkload(wl)
    for mode in (0, 1, 2):
        assert csa2.csa2_layer_workspace_size(mode, dw.batch) <= SCRATCH_BYTES
    want = _run(dw, use_noalloc=False)
    _same(_run(dw, use_noalloc=True), want, "first pass")
    # an unrelated workload (other seed, shapes, layer pattern) through the array
    other = DeviceWorkload(W.Workload("noalloc_other", 9191, 2, [9000, 30000], 1,
                                      ["full", "reindex", "reuse"], planted_blocks=2))
    _run(other, use_noalloc=True)
    _same(_run(dw, use_noalloc=True), want, "after another workload")
    assert int(dw.cache.status[0]) == 0 and int(other.cache.status[0]) == 0


def test_noalloc_refuses_early_all():
    """csa2_layer_noalloc cannot give a call a workspace of its own, so it
    refuses csa2.ATTN_EARLY_ALL before touching the device."""
    lib = csa2.load()
    P = ctypes.c_void_p(1 << 12)
    b = csa2.Batch(8, 1, 1, 0, 4096, P, P)
    s = csa2.Swa(P, P, 128, csa2.ATTN_EARLY_INPUTS | csa2.ATTN_EARLY_ALL, None, None, None, 0.0, 0)
    io = csa2.LayerIO(P, P, P, s, 1.0, 0, P, P, P, P, P, None, None)
    assert lib.csa2_layer_noalloc(2, None, ctypes.byref(b), ctypes.byref(io), None) == -3


def test_noalloc_refuses_work_beyond_its_scratch():
    lib = csa2.load()
    big = csa2.Batch(8, 1, 1, 0, 1 << 20, None, None)           # a Full layer over 8 x 1M entries
    assert lib.csa2_layer_workspace_size(0, ctypes.byref(big)) > SCRATCH_BYTES
    cache, io = csa2.Cache(), csa2.LayerIO()
    st = lib.csa2_layer_noalloc(0, ctypes.byref(cache), ctypes.byref(big), ctypes.byref(io), None)
    assert st == -5                                              # CSA2_ERR_WORKSPACE, nothing launched
    # a Reindex layer of 8 rows needs the attention's scratch and its rescored pools
    # (about 5.8 MB): past the size check, it fails on the NULL cache, still before
    # any launch
    st = lib.csa2_layer_noalloc(1, ctypes.byref(cache), ctypes.byref(big), ctypes.byref(io), None)
    assert st == -1                                              # CSA2_ERR_NULL from csa2_layer's checks
