"""Device-side set-up and layer driver for a synthetic CSA2 workload.

Builds the paged cache with the library's own quantisers (csa2_quant_mxfp4 /
csa2_quant_fp8 / csa2_compress) from the seeded generator, allocates the
per-layer inputs, window rings, selection state, outputs and workspace, and
runs the decoder (or encoder) layer pattern through csa2_layer.  Python here
only allocates device memory and marshals arguments; every step of the path
runs in the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

from . import csa2, synth
from .workloads import Workload, T_C, T_IK, T_Q, T_QI, T_SWA, T_W, T_Z

_CHUNK = 1 << 16   # entries per cache-building chunk


def _dev_normal_bf16(stream, start, count, dev, sigma=1.0):
    return synth.normal_bf16_torch(stream, start, count, dev, sigma)


class DeviceWorkload:
    def __init__(self, wl: Workload, device="cuda", build_cache=True, layers=None):
        self.wl = wl
        self.dev = torch.device(device)
        self.rows = wl.batch * wl.nq
        self.layers = list(range(len(wl.layers))) if layers is None else list(layers)
        bt = torch.from_numpy(wl.block_table())
        self.cache = csa2.PagedCache(wl.total_pages, bt, self.dev, kv_format=wl.kv_format)
        self.n_entries = torch.tensor([wl.entries(b) for b in range(wl.batch)], dtype=torch.int64, device=self.dev)
        self.q_pos = torch.from_numpy(np.concatenate([wl.q_pos(b) for b in range(wl.batch)])).to(self.dev)
        self.batch = csa2.batch_struct(self.n_entries, self.q_pos, wl.nq, wl.m, wl.max_entries)
        self.cstruct = self.cache.struct()
        if build_cache:
            self.build_cache()
        self._alloc_layers()

    # ------------------------------------------------------------ cache
    def entry_slots(self, b: int, e0: int, e1: int) -> torch.Tensor:
        e = torch.arange(e0, e1, dtype=torch.int64, device=self.dev)
        return self.cache.slots(b, e)

    def build_cache(self):
        wl, dev = self.wl, self.dev
        for b in range(wl.batch):
            E = wl.entries(b)
            pos, rows = wl.planted_rows(b)
            pos_d = torch.from_numpy(pos).to(dev)
            rows_d = torch.from_numpy(rows).to(dev)
            for e0 in range(0, E, _CHUNK):
                e1 = min(E, e0 + _CHUNK)
                slots = self.entry_slots(b, e0, e1)
                # main KV: m = 1 -> the entry is C itself; m > 1 -> the compressor
                if wl.m == 1:
                    x = _dev_normal_bf16(wl._sid(T_C, b), e0 * 512, (e1 - e0) * 512, dev).float().view(e1 - e0, 512)
                else:
                    x = self.compress_tokens(b, e0 * wl.m, e1 * wl.m)
                quant = csa2.csa2_quant_fp4_e4m3 if wl.kv_format == csa2.KV_FP4_E4M3 else csa2.csa2_quant_mxfp4
                quant(x, self.cache.kv_codes, self.cache.kv_scales, slots=slots, status=self.cache.status)
                # indexer keys with planted rows
                k = synth.normal_f32_torch(wl._sid(T_IK, b), e0 * 128, (e1 - e0) * 128, dev).view(e1 - e0, 128)
                sel = (pos_d >= e0) & (pos_d < e1)
                if bool(sel.any()):
                    k[pos_d[sel] - e0] = rows_d[sel]
                csa2.csa2_quant_fp8(k, self.cache.ik_codes, self.cache.ik_scales, slots=slots,
                                    status=self.cache.status)

    def compress_tokens(self, b: int, t0: int, t1: int) -> torch.Tensor:
        """Compressor over tokens [t0, t1) of sequence b (t0, t1 multiples of m)."""
        wl, dev = self.wl, self.dev
        C = _dev_normal_bf16(wl._sid(T_C, b), t0 * 512, (t1 - t0) * 512, dev).view(t1 - t0, 512)
        Z = _dev_normal_bf16(wl._sid(T_Z, b), t0 * 512, (t1 - t0) * 512, dev).view(t1 - t0, 512)
        bias = torch.from_numpy(wl.bias()).to(dev)
        out = torch.empty(((t1 - t0) // wl.m, 512), dtype=torch.float32, device=dev)
        csa2.csa2_compress(C, Z, bias, wl.m, out)
        return out

    # ------------------------------------------------------------ layers
    def _alloc_layers(self):
        wl, dev, R = self.wl, self.dev, self.rows
        self.q, self.qi, self.w, self.swa_codes, self.swa_scales = {}, {}, {}, {}, {}
        for l in self.layers:
            self.q[l] = self._layer_q(l)
            if wl.layers[l] != "reuse":
                self.qi[l] = torch.from_numpy(
                    np.concatenate([wl.qi_bits(l, b) for b in range(wl.batch)]).view(np.int16)).to(dev).view(torch.bfloat16) \
                    if wl.nq * wl.batch <= 4096 else self._layer_qi_device(l)
                self.w[l] = self._layer_w(l)
            self._fill_swa(l)
        self.idx = torch.full((R, csa2.TOPK), -1, dtype=torch.int32, device=dev)
        self.pool = torch.full((R, csa2.POOL_MAX), -1, dtype=torch.int32, device=dev)
        self.pool_len = torch.zeros((R,), dtype=torch.int32, device=dev)
        # attention options passed to every layer call (csa2.swa_struct keywords:
        # sink, rope_base, flags); none by default
        self.attn_options = {}
        self.layer_flags = 0             # csa2.LAYER_* bits for every layer call
        # Reuse layers load their keys while the previous layer finishes
        # (csa2.ATTN_EARLY_INPUTS): the layers are called one after the other
        self.early_inputs = True
        # ... and with early_all their whole attention (csa2.ATTN_EARLY_ALL): q and
        # the window rows are in place before the layers run, and a Reuse layer
        # takes the workspace the previous call did not use
        self.early_all = False
        self.workspace_alt = None
        self._last_ws = None
        self.o = {l: torch.empty((R, 64, 512), dtype=torch.float32, device=dev) for l in self.layers}
        self.lse = {l: torch.empty((R, 64), dtype=torch.float32, device=dev) for l in self.layers}
        ws = max(csa2.csa2_layer_workspace_size(m, self.batch) for m in (0, 1, 2))
        self.workspace = torch.empty((ws + 255) // 256 * 256, dtype=torch.uint8, device=dev)
        self.dummy_qi = torch.zeros((R, 32, 128), dtype=torch.bfloat16, device=dev)
        self.dummy_w = torch.zeros((R, 32), dtype=torch.float32, device=dev)

    def _layer_q(self, l):
        wl, dev = self.wl, self.dev
        parts = [_dev_normal_bf16(wl._sid(T_Q, b, l), 0, wl.nq * 32768, dev, sigma=512 ** -0.5)
                 for b in range(wl.batch)]
        return torch.cat(parts).view(self.rows, 64, 512)

    def _layer_qi_device(self, l):
        wl, dev = self.wl, self.dev
        assert wl.layers[l] == "full"
        parts = [_dev_normal_bf16(wl._sid(T_QI, b, l), 0, wl.nq * 4096, dev) for b in range(wl.batch)]
        return torch.cat(parts).view(self.rows, 32, 128)

    def _layer_w(self, l):
        wl, dev = self.wl, self.dev
        parts = [synth.uniform_f32_torch(wl._sid(T_W, b, l), 0, wl.nq * 32, dev) for b in range(wl.batch)]
        return torch.cat(parts).view(self.rows, 32)

    def _fill_swa(self, l):
        wl, dev = self.wl, self.dev
        Rr = wl.swa_rows
        codes = torch.zeros((wl.batch, Rr, 512), dtype=torch.uint8, device=dev)
        scales = torch.ones((wl.batch, Rr), dtype=torch.float32, device=dev)
        for b in range(wl.batch):
            t0, t1 = wl.swa_tokens(b)
            x = _dev_normal_bf16(wl._sid(T_SWA, b, l), t0 * 512, (t1 - t0) * 512, dev).float().view(t1 - t0, 512)
            rows = torch.arange(t0, t1, dtype=torch.int64, device=dev) % Rr + b * Rr
            csa2.csa2_quant_fp8(x, codes.view(-1, 512), scales.view(-1), slots=rows)
        self.swa_codes[l] = codes
        self.swa_scales[l] = scales

    def swa(self, l, new_rows=None) -> csa2.Swa:
        opts = dict(self.attn_options)
        if self.early_inputs and self.wl.layers[l] == "reuse":
            # every layer call follows the previous one on the stream (run / run_layer in order)
            opts["flags"] = opts.get("flags", 0) | csa2.ATTN_EARLY_INPUTS
            if self.early_all:
                opts["flags"] |= csa2.ATTN_EARLY_ALL
        return csa2.swa_struct(self.swa_codes[l], self.swa_scales[l], new_rows=new_rows, **opts)

    def swa_new_rows(self, l) -> torch.Tensor:
        """fp32 [B][512]: the window row of each sequence's decode token (nq = 1)."""
        wl, dev = self.wl, self.dev
        assert wl.nq == 1
        return torch.cat([_dev_normal_bf16(wl._sid(T_SWA, b, l), int(wl.q_pos(b)[0]) * 512, 512, dev).float()
                          for b in range(wl.batch)]).view(wl.batch, 512)

    def io(self, l, prof=None, new_rows=None) -> csa2.LayerIO:
        qi = self.qi.get(l, self.dummy_qi)
        w = self.w.get(l, self.dummy_w)
        return csa2.layer_io(self.q[l], qi, w, self.swa(l, new_rows), 1.0, self.idx, self.pool, self.pool_len,
                             self.o[l], self.lse[l], prof=prof, flags=self.layer_flags)

    def run_layer(self, l, stream=None, prof=None, new_rows=None):
        """new_rows: optional window rows of the decode tokens, quantised into the
        ring by the layer call itself (see csa2_swa.new_rows)."""
        mode = csa2.MODES[self.wl.layers[l]]
        ws = self.workspace
        if self.early_inputs and self.early_all and self.wl.layers[l] == "reuse":
            if self.workspace_alt is None:
                n = csa2.csa2_layer_workspace_size(csa2.MODES["reuse"], self.batch)
                self.workspace_alt = torch.empty((n + 255) // 256 * 256, dtype=torch.uint8, device=self.dev)
            if self._last_ws is self.workspace:
                ws = self.workspace_alt
        self._last_ws = ws
        csa2.csa2_layer(mode, self.cstruct, self.batch, self.io(l, prof, new_rows), ws, stream=stream)

    def run(self, stream=None, on_layer=None):
        for l in self.layers:
            self.run_layer(l, stream)
            if on_layer is not None:
                on_layer(l)
