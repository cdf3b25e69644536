"""Oracle-side expected results for a workload (host only).

Regenerates a sequence's inputs from the seeded generator and runs the CPU
oracle step by step in the pages' order.  Nothing here reads any output of
the CUDA path.
"""
from __future__ import annotations

import numpy as np

import oracle
from compressed_sparse_attention_layer_gb300.workloads import Workload


class SeqOracle:
    """Oracle state of one sequence b of a workload."""

    def __init__(self, wl: Workload, b: int):
        self.wl, self.b = wl, b
        self.E = wl.entries(b)
        self.planted = wl.planted_rows(b)
        self._ik = None

    # indexer keys of every entry (FP8 by the oracle's quantiser)
    def ik(self):
        if self._ik is None:
            self._ik = oracle.quant_fp8(self.wl.ik_src(self.b, 0, self.E, planted=self.planted))
        return self._ik

    # main-KV entries at given positions (FP4 in the workload's format, by the oracle's quantiser)
    def kv(self, positions):
        wl, b = self.wl, self.b
        pos = np.asarray(positions, np.int64)
        if wl.m == 1:
            src = np.concatenate([wl.kv_src(b, int(p), int(p) + 1) for p in pos]) if pos.size else np.zeros((0, 512), np.float32)
        else:
            bias = wl.bias()
            rows = []
            for p in pos:
                C, Z = wl.cz_bits(b, int(p) * wl.m, (int(p) + 1) * wl.m)
                rows.append(oracle.compress(C, Z, bias, wl.m))
            src = np.concatenate(rows) if rows else np.zeros((0, 512), np.float32)
        return oracle.KV_FORMATS[wl.kv_format][0](src)

    # the layer's window ring as the oracle quantises it
    def swa_ring(self, layer):
        wl, b = self.wl, self.b
        R = wl.swa_rows
        t0, t1 = wl.swa_tokens(b)
        codes = np.zeros((R, 512), np.uint8)
        scales = np.ones((R,), np.float32)
        c, s = oracle.quant_fp8(wl.swa_src(layer, b, t0, t1))
        rows = np.arange(t0, t1) % R
        codes[rows] = c
        scales[rows] = s
        return codes, scales

    def visible(self, i):
        t = int(self.wl.q_pos(self.b)[i])
        return t, oracle.n_visible(t, self.wl.m, self.E)

    def full(self, layer, i):
        """(idx, pool, scores) of query i at a Full layer."""
        t, nvis = self.visible(i)
        qi = self.wl.qi_bits(layer, self.b, [i])[0]
        w = self.wl.w(layer, self.b, [i])[0]
        codes, scales = self.ik()
        return oracle.full_select(qi, w, codes, scales, nvis)

    def reindex(self, layer, i, pool):
        qi = self.wl.qi_bits(layer, self.b, [i])[0]
        w = self.wl.w(layer, self.b, [i])[0]
        codes, scales = self.ik()
        return oracle.reindex_select(qi, w, codes, scales, pool)

    def scores(self, layer, i, positions):
        qi = self.wl.qi_bits(layer, self.b, [i])[0]
        w = self.wl.w(layer, self.b, [i])[0]
        codes, scales = self.ik()
        return oracle.index_scores(qi, w, codes, scales, positions=np.asarray(positions, np.int32))

    def attention(self, layer, i, idx, ring=None, sink=None, rope_base=0.0, dedup=False, q_bits=None):
        """o, lse of query i over the selected entries idx and its window; sink,
        rope_base and dedup (drop selected entries that are window rows) as in
        oracle.attention / oracle.dedup_selection; q_bits: the query's bf16 bits
        [64][512] in place of the workload's own."""
        t, _ = self.visible(i)
        sel = np.asarray(idx, np.int64)
        sel = sel[sel >= 0]
        if dedup:
            sel = oracle.dedup_selection(sel, t, self.wl.m)
        kvc, kvs = self.kv(sel)
        swc, sws = ring if ring is not None else self.swa_ring(layer)
        keys = oracle.attention_keys(kvc, kvs, np.arange(sel.size, dtype=np.int32), swc, sws, t,
                                     kv_format=self.wl.kv_format)
        q = self.wl.q_bits(layer, self.b, [i])[0] if q_bits is None else q_bits
        return oracle.attention(q, 1.0, keys, sink=sink, rope_base=rope_base, t=t)

    def layers(self, i, upto=None):
        """Expected (idx, o, lse) of query i for each layer, run in order."""
        out = []
        idx = pool = None
        for l, mode in enumerate(self.wl.layers[:upto]):
            if mode == "full":
                idx, pool, _ = self.full(l, i)
            elif mode == "reindex":
                idx, _ = self.reindex(l, i, pool)
            o, lse = self.attention(l, i, idx)
            out.append((idx.copy(), o, lse))
        return out


def attn_close(o, lse, o_ref, lse_ref, max_abs=2e-3, rel_l2=1e-3):
    """Attention tolerance: max-abs 2e-3 and rel-L2 1e-3 on o; lse to 1e-4."""
    o = np.asarray(o, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    err = np.abs(o - o_ref).max()
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    lerr = np.abs(np.asarray(lse, np.float64) - np.asarray(lse_ref, np.float64)).max()
    return err <= max_abs and rel <= rel_l2 and lerr <= 1e-4 * max(1.0, np.abs(lse_ref).max()), (err, rel, lerr)


def topk_valid(sel, scores_of, kth, overlap_ref, min_overlap=0.995):
    """Top-K rule: every selected index scores >= the oracle's k-th score minus
    1e-3 |score|, and at least 99.5% of the set overlaps the oracle's."""
    sel = np.asarray(sel)
    sel = sel[sel >= 0]
    ref = np.asarray(overlap_ref)
    ref = ref[ref >= 0]
    s = scores_of(sel)
    ok_valid = bool(np.all(s >= kth - 1e-3 * np.abs(kth)))
    ov = np.intersect1d(sel, ref).size / max(ref.size, 1)
    return ok_valid and ov >= min_overlap and sel.size == ref.size, (ok_valid, ov, sel.size, ref.size)
