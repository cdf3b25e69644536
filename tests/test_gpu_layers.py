"""Whole layers through csa2_layer against the oracle (needs a GPU).

Rules (from the task's correctness bar): Reuse propagation bit-exact; Top-K
valid (every selected index scores >= the oracle's k-th score - 1e-3|score|)
with >= 99.5% overlap; attention within max-abs 2e-3 / rel-L2 1e-3 given the
same indices (checked whenever the GPU and oracle sets agree, which the
planted workloads make the common case).
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_layer_gb300 import workloads as W
from compressed_sparse_attention_layer_gb300.device import DeviceWorkload
from tests.reference import SeqOracle, attn_close, topk_valid

pytestmark = pytest.mark.gpu


def _check_sequence(dw, b, i=0, check_attn_when_equal=True):
    wl = dw.wl
    so = SeqOracle(wl, b)
    r = b * wl.nq + i
    ring = {}
    pool_ref = None
    idx_ref = None
    for l, mode in enumerate(wl.layers):
        got_idx = dw.hist_idx[l][r]
        if mode == "full":
            idx_ref, pool_ref, scores = so.full(l, i)
            kth = np.sort(scores[pool_ref])[::-1][min(511, pool_ref.size - 1)]
            ok, info = topk_valid(got_idx, lambda s: scores[s], kth, idx_ref)
            assert ok, (l, mode, info)
            # pool: same size; the planted blocks are in it
            assert dw.hist_pool_len[l][r] == pool_ref.size
        elif mode == "reindex":
            idx_ref, ps = so.reindex(l, i, pool_ref)
            kth = np.sort(ps)[::-1][min(511, ps.size - 1)]
            ok, info = topk_valid(got_idx, lambda s: so.scores(l, i, s), kth, idx_ref)
            assert ok, (l, mode, info)
        else:
            assert np.array_equal(got_idx, dw.hist_idx[l - 1][r]), (l, "reuse must copy bit-exactly")
        sel = got_idx if check_attn_when_equal else idx_ref
        if np.array_equal(np.sort(got_idx), np.sort(idx_ref)):
            o_ref, lse_ref = so.attention(l, i, idx_ref)
            ok, info = attn_close(dw.o[l][r].cpu().numpy(), dw.lse[l][r].cpu().numpy(), o_ref, lse_ref)
            assert ok, (l, mode, info)


def _run_recording(dw):
    dw.hist_idx, dw.hist_pool_len = {}, {}

    def rec(l):
        dw.hist_idx[l] = dw.idx.cpu().numpy().copy()
        dw.hist_pool_len[l] = dw.pool_len.cpu().numpy().copy()

    dw.run(on_layer=rec)
    torch.cuda.synchronize()
    assert int(dw.cache.status[0]) == 0


def test_layer_decode_small():
    dw = DeviceWorkload(W.decode_small())
    _run_recording(dw)
    _check_sequence(dw, 0)
    # 4,096 entries: 512 blocks, the pool is every position
    assert dw.hist_pool_len[0][0] == 4096


@pytest.mark.parametrize("tokens", [1, 7, 64, 129, 512, 1000])
def test_layer_tiny_contexts(tokens):
    """Short sequences: Top-K covers every visible entry (the dense case)."""
    wl = W.Workload("tiny", 77 + tokens, 3, [tokens, max(1, tokens // 2), tokens + 3], 1,
                    ["full", "reuse", "reindex", "reuse"])
    dw = DeviceWorkload(wl)
    _run_recording(dw)
    for b in range(wl.batch):
        so = SeqOracle(wl, b)
        if wl.entries(b) <= 512:
            for l in range(len(wl.layers)):
                got = dw.hist_idx[l][b]
                assert np.array_equal(np.sort(got[got >= 0]), np.arange(wl.entries(b)))
                o_ref, lse_ref = so.attention(l, 0, got)
                ok, info = attn_close(dw.o[l][b].cpu().numpy(), dw.lse[l][b].cpu().numpy(), o_ref, lse_ref)
                assert ok, (b, l, info)
        else:
            _check_sequence(dw, b)


def test_layer_decode_group_full_size():
    """64 x 32,768 tokens, random page permutation, 16 planted blocks each;
    Full + 3 Reuse, Reindex + 3 Reuse.  Four sequences checked end to end,
    the planted set checked on all 64."""
    wl = W.decode_group()
    dw = DeviceWorkload(wl)
    _run_recording(dw)
    for b in (0, 17, 40, 63):
        _check_sequence(dw, b)
    for b in range(wl.batch):
        assert np.isin(wl.planted_positions(b), dw.hist_idx[0][b]).all()
