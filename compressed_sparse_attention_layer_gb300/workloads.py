"""The five synthetic CSA2 workloads and their seeded inputs.

Each workload is described by plain numbers (batch, context lengths, m,
layer modes, planted blocks).  Its tensors come from the counter-based
generator in :mod:`synth`, so any slice can be regenerated on the host for
the oracle or on the device for the CUDA path, bit for bit.  Nothing here
computes any part of the method: the planted keys are input construction.

Workloads (sizes from the task's configurations):
  decode_small   1 x 4,096 tokens, one Full layer, Top-512 over 512 blocks.
  decode_group   64 x 32,768 tokens, paged with a random page permutation,
                 16 planted blocks per sequence, layers Full + 3 Reuse,
                 Reindex + 3 Reuse.
  prefill        8,192 new tokens after a 65,536-token prefix, m = 2
                 (36,864 entries), causal, Full + 5 Reuse.
  decode_1m      8 x 1,048,576 tokens, 64 planted blocks per sequence, the
                 20-layer decoder pattern (Full + 3 Reuse, 4 x (Reindex + 3 Reuse)).
  decode_ragged  128 sequences, log-uniform lengths in [4,096, 1,048,576],
                 the 20-layer decoder pattern, per-layer seeds.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List

import numpy as np

from . import synth

DECODER_STACK = ["full", "reuse", "reuse", "reuse"] + ["reindex", "reuse", "reuse", "reuse"] * 4
DECODER_GROUP_PAIR = ["full", "reuse", "reuse", "reuse", "reindex", "reuse", "reuse", "reuse"]
ENCODER_GROUP = ["full"] + ["reuse"] * 5

# tensor ids of the generator streams
T_C, T_Z, T_BIAS, T_IK, T_Q, T_QI, T_W, T_SWA, T_PLANT, T_FRESH, T_QI_FRESH, T_PAGES, T_LEN = range(1, 14)

PAGE = 64
W = 128


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    batch: int
    tokens: List[int]            # context tokens N_b (decode: includes the current token)
    m: int
    layers: List[str]
    planted_blocks: int = 0
    nq: int = 1                  # query tokens per sequence
    prefill_new: int = 0         # prefill: the last prefill_new tokens are the queries
    page_permute: bool = True
    swa_rows: int = W
    kv_format: int = 0           # main KV: 0 MXFP4 (32-element blocks, E8M0), 1 FP4 with E4M3 per 16

    # ------------------------------------------------------------ geometry
    def entries(self, b: int) -> int:
        return self.tokens[b] // self.m

    @property
    def max_entries(self) -> int:
        return max(self.entries(b) for b in range(self.batch))

    def pages(self, b: int) -> int:
        return (self.entries(b) + PAGE - 1) // PAGE

    @property
    def max_pages(self) -> int:
        return max(self.pages(b) for b in range(self.batch))

    @property
    def total_pages(self) -> int:
        return sum(self.pages(b) for b in range(self.batch))

    def q_pos(self, b: int) -> np.ndarray:
        N = self.tokens[b]
        if self.prefill_new:
            return np.arange(N - self.prefill_new, N, dtype=np.int64)
        return np.array([N - 1], dtype=np.int64)

    def block_table(self) -> np.ndarray:
        """[batch][max_pages] page ids; unused tail entries are -1."""
        tot = self.total_pages
        if self.page_permute:
            perm = np.random.default_rng(synth.stream_id(self.seed, T_PAGES)).permutation(tot)
        else:
            perm = np.arange(tot)
        bt = np.full((self.batch, self.max_pages), -1, np.int32)
        off = 0
        for b in range(self.batch):
            n = self.pages(b)
            bt[b, :n] = perm[off:off + n]
            off += n
        return bt

    def first_full_layer(self, layer: int) -> int:
        """Index of the most recent Full layer at or before `layer`."""
        for l in range(layer, -1, -1):
            if self.layers[l] == "full":
                return l
        raise ValueError("no Full layer before this one")

    # ------------------------------------------------------------ per-layer inputs (host)
    def _sid(self, tensor: int, b: int = 0, layer: int = 0) -> int:
        return synth.stream_id(self.seed, tensor, b, layer)

    def q_bits(self, layer: int, b: int, qrows=None) -> np.ndarray:
        """bf16 [nq_sel, 64, 512] attention queries, N(0,1)/sqrt(512)."""
        rows = np.arange(self.nq) if qrows is None else np.asarray(qrows)
        out = np.empty((rows.size, 64 * 512), np.uint16)
        for k, i in enumerate(rows):
            out[k] = synth.normal_bf16(self._sid(T_Q, b, layer), int(i) * 32768, 32768, sigma=512 ** -0.5)
        return out.reshape(rows.size, 64, 512)

    def qi_bits(self, layer: int, b: int, qrows=None) -> np.ndarray:
        """bf16 [nq_sel, 32, 128] indexer queries.  A Full layer draws N(0,1); a
        Reindex layer mixes 0.8 x the Full layer's query with 0.6 x a fresh
        draw (so the pool stays relevant), rounded once to bf16."""
        rows = np.arange(self.nq) if qrows is None else np.asarray(qrows)
        out = np.empty((rows.size, 4096), np.uint16)
        mode = self.layers[layer]
        for k, i in enumerate(rows):
            if mode == "full" or mode == "reuse":
                out[k] = synth.normal_bf16(self._sid(T_QI, b, layer), int(i) * 4096, 4096)
            else:
                lf = self.first_full_layer(layer)
                base = synth.bf16_bits_to_f32(synth.normal_bf16(self._sid(T_QI, b, lf), int(i) * 4096, 4096))
                fresh = synth.bf16_bits_to_f32(synth.normal_bf16(self._sid(T_QI_FRESH, b, layer), int(i) * 4096, 4096))
                mix = (0.8 * base.astype(np.float64) + 0.6 * fresh.astype(np.float64)).astype(np.float32)
                out[k] = synth._f32_to_bf16_bits(mix)
        return out.reshape(rows.size, 32, 128)

    def w(self, layer: int, b: int, qrows=None) -> np.ndarray:
        rows = np.arange(self.nq) if qrows is None else np.asarray(qrows)
        out = np.empty((rows.size, 32), np.float32)
        lw = layer if self.layers[layer] != "reuse" else self.first_full_layer(layer)
        for k, i in enumerate(rows):
            out[k] = synth.uniform_f32(self._sid(T_W, b, lw), int(i) * 32, 32)
        return out

    def swa_src(self, layer: int, b: int, t0: int, t1: int) -> np.ndarray:
        """fp32 [t1-t0, 512] window-KV source of tokens [t0, t1) (bf16 values)."""
        bits = synth.normal_bf16(self._sid(T_SWA, b, layer), t0 * 512, (t1 - t0) * 512)
        return synth.bf16_bits_to_f32(bits).reshape(t1 - t0, 512)

    def swa_tokens(self, b: int):
        """Tokens whose window rows the queries need: [max(0, t_min-127), t_max]."""
        qp = self.q_pos(b)
        return max(0, int(qp.min()) - (W - 1)), int(qp.max()) + 1

    # ------------------------------------------------------------ main KV source
    def kv_src(self, b: int, e0: int, e1: int) -> np.ndarray:
        """m = 1: fp32 [e1-e0, 512] entries (the compressor is the identity)."""
        assert self.m == 1
        bits = synth.normal_bf16(self._sid(T_C, b), e0 * 512, (e1 - e0) * 512)
        return synth.bf16_bits_to_f32(bits).reshape(e1 - e0, 512)

    def cz_bits(self, b: int, t0: int, t1: int):
        """m > 1: bf16 patterns of C and Z for tokens [t0, t1)."""
        C = synth.normal_bf16(self._sid(T_C, b), t0 * 512, (t1 - t0) * 512).reshape(t1 - t0, 512)
        Z = synth.normal_bf16(self._sid(T_Z, b), t0 * 512, (t1 - t0) * 512).reshape(t1 - t0, 512)
        return C, Z

    def bias(self) -> np.ndarray:
        """[m, 512] learned-bias stand-in, N(0, 0.1^2)."""
        return synth.normal_f32(self._sid(T_BIAS), 0, self.m * 512, sigma=0.1).reshape(self.m, 512)

    # ------------------------------------------------------------ indexer keys
    def planted(self, b: int) -> np.ndarray:
        """Sorted ids of the planted blocks of sequence b (outside the window)."""
        if not self.planted_blocks:
            return np.zeros((0,), np.int64)
        eligible = (self.entries(b) - W) // 8
        rng = np.random.default_rng(self._sid(T_PLANT, b))
        return np.sort(rng.choice(eligible, self.planted_blocks, replace=False)).astype(np.int64)

    def planted_positions(self, b: int) -> np.ndarray:
        blk = self.planted(b)
        return (blk[:, None] * 8 + np.arange(8)[None]).reshape(-1)

    def _ik_raw(self, b: int, e0: int, e1: int) -> np.ndarray:
        return synth.normal_f32(self._sid(T_IK, b), e0 * 128, (e1 - e0) * 128).reshape(e1 - e0, 128)

    def planted_rows(self, b: int):
        """(positions, fp32 [n, 128]) keys planted at cosine 0.6 with the
        direction of sum_h w_h q_h of the first Full layer's query:
        k = |g| (0.6 u + 0.8 v), g the original N(0, I) key, v a fresh unit
        vector orthogonal to u."""
        pos = self.planted_positions(b)
        if pos.size == 0:
            return pos, np.zeros((0, 128), np.float32)
        lf = self.layers.index("full")
        qi = synth.bf16_bits_to_f32(self.qi_bits(lf, b, [0])[0]).astype(np.float64)
        w = self.w(lf, b, [0])[0].astype(np.float64)
        u = (w[:, None] * qi).sum(axis=0)
        u /= np.linalg.norm(u)
        rows = np.empty((pos.size, 128), np.float32)
        for k, p in enumerate(pos):
            g = self._ik_raw(b, int(p), int(p) + 1)[0].astype(np.float64)
            f = synth.normal_f32(self._sid(T_FRESH, b), int(p) * 128, 128).astype(np.float64)
            v = f - (f @ u) * u
            v /= np.linalg.norm(v)
            rows[k] = (np.linalg.norm(g) * (0.6 * u + 0.8 * v)).astype(np.float32)
        return pos, rows

    def ik_src(self, b: int, e0: int, e1: int, planted=None) -> np.ndarray:
        """fp32 [e1-e0, 128] indexer-key source with the planted rows in place."""
        x = self._ik_raw(b, e0, e1)
        pos, rows = planted if planted is not None else self.planted_rows(b)
        sel = (pos >= e0) & (pos < e1)
        x[pos[sel] - e0] = rows[sel]
        return x


# ---------------------------------------------------------------- the five workloads
def decode_small(seed: int = 1000) -> Workload:
    return Workload("decode_small", seed, 1, [4096], 1, ["full"], page_permute=False)


def decode_group(seed: int = 2000, batch: int = 64, tokens: int = 32768) -> Workload:
    return Workload("decode_group", seed, batch, [tokens] * batch, 1, list(DECODER_GROUP_PAIR), planted_blocks=16)


def prefill(seed: int = 3000, prefix: int = 65536, new: int = 8192) -> Workload:
    n = prefix + new
    return Workload("prefill", seed, 1, [n], 2, list(ENCODER_GROUP), nq=new, prefill_new=new,
                    swa_rows=new + W)


def decode_1m(seed: int = 4000, batch: int = 8, tokens: int = 1 << 20, layers=None, kv_format: int = 0) -> Workload:
    return Workload("decode_1m", seed, batch, [tokens] * batch, 1, list(layers or DECODER_STACK), planted_blocks=64,
                    kv_format=kv_format)


def decode_multi(seed: int = 6000, batch: int = 8, tokens: int = 1 << 20, q: int = 4, layers=None,
                 planted_blocks: int = 64) -> Workload:
    """Multi-token decode (draft tokens verified in one step): the last q
    tokens of each sequence are queries, each with its own causal range."""
    return Workload("decode_multi", seed, batch, [tokens] * batch, 1, list(layers or DECODER_STACK),
                    planted_blocks=planted_blocks, nq=q, prefill_new=q, swa_rows=W + q)


def ragged_lengths(seed: int, batch: int, lo: int = 4096, hi: int = 1 << 20) -> List[int]:
    rng = np.random.default_rng(synth.stream_id(seed, T_LEN))
    return [int(math.floor(math.exp(v))) for v in rng.uniform(math.log(lo), math.log(hi), batch)]


def decode_ragged(seed: int = 5000, batch: int = 128) -> Workload:
    return Workload("decode_ragged", seed, batch, ragged_lengths(seed, batch), 1, list(DECODER_STACK))


WORKLOADS = {"decode_small": decode_small, "decode_group": decode_group, "prefill": prefill,
             "decode_1m": decode_1m, "decode_ragged": decode_ragged}
