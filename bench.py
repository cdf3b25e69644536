#!/usr/bin/env python
"""CSA2 decode benchmark: query-tokens/s at 1,048,576-token context, batch 8.

One step = one decode token for each of the 8 sequences through the whole
hot path: the new token's entry is compressed (m = 1) and quantised into the
paged cache (MXFP4 main KV, FP8 indexer key), then the 20-layer decoder
pattern runs (Full + 3 Reuse, 4 x (Reindex + 3 Reuse)) through csa2_layer,
whose attention call also quantises the layer's FP8 window row of the new
token into its ring.  The step is captured once as a CUDA graph and replayed.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tokens/s at 1M ctx (batch 8); % of HBM roofline"
UNIT = "query-tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--batch", type=int, default=8)
    p.add_argument("--tokens", type=int, default=1 << 20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--kv-format", type=int, default=0, choices=[0, 1],
                   help="main KV: 0 MXFP4 (32-element blocks, E8M0), 1 FP4 with an E4M3 scale per 16 elements")
    p.add_argument("--workload", default="decode_1m",
                   choices=["decode_1m", "decode_small", "decode_group", "decode_ragged", "prefill", "norm_rope"],
                   help="decode_1m (default: the headline, batch 8 x 1M tokens); the other four synthetic "
                        "workloads run the same step for their own shapes (prefill: one 8,192-token chunk); "
                        "norm_rope times the input prologue alone (RMSNorm + RoPE of a prefill chunk's queries)")
    p.add_argument("--bf16-scores", action="store_true",
                   help="Full and Reindex layers select on bf16-rounded index scores (csa2.LAYER_SCORES_BF16)")
    p.add_argument("--e4m3-query", action="store_true",
                   help="the Full layer's scan with one e4m3 query part per head (csa2.LAYER_INDEX_E4M3_QUERY)")
    p.add_argument("--attn-schedule", default="auto", choices=["auto", "chunks", "rows"],
                   help="attention schedule (csa2.ATTN_SCHEDULE_*): one cluster per (row, key chunk) and a "
                        "merge, or persistent clusters over whole rows; auto picks by the number of rows")
    p.add_argument("--no-early-all", action="store_true",
                   help="Reuse layers wait for the previous layer before their attention's products "
                        "(csa2.ATTN_EARLY_INPUTS only, instead of csa2.ATTN_EARLY_ALL)")
    p.add_argument("--queries", type=int, default=1,
                   help="query tokens per sequence per step (>1: a multi-token decode step, e.g. draft "
                        "tokens verified together; the Full layer's scan serves them from one read)")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------- ranks
def rank_seed(rank: int) -> int:
    """Each rank decodes its own batch of sequences (weak scaling): its own seed."""
    return 4000 + 7919 * rank


def reduce_max(x: float, device, world: int) -> float:
    """The maximum of x over the ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, batch: int, steps: int, seconds: float) -> float:
    """Query tokens per second of the whole job: every rank decodes batch tokens per step."""
    return world * batch * steps / seconds


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the decode step
class DecodeStep:
    """Device state and the launch sequence of one decode step."""

    def __init__(self, batch, tokens, seed, device, kv_format=0, queries=1, workload="decode_1m", early_all=True):
        import numpy as np
        import torch
        from compressed_sparse_attention_layer_gb300 import csa2, synth
        from compressed_sparse_attention_layer_gb300 import workloads as W
        from compressed_sparse_attention_layer_gb300.device import DeviceWorkload

        self.torch, self.csa2 = torch, csa2
        if workload == "decode_1m" and queries == 1:
            self.wl = W.decode_1m(seed=seed, batch=batch, tokens=tokens, kv_format=kv_format)
        elif workload == "decode_1m":
            self.wl = W.decode_multi(seed=seed, batch=batch, tokens=tokens, q=queries)
        else:
            make = {"decode_small": W.decode_small, "decode_group": W.decode_group,
                    "decode_ragged": W.decode_ragged, "prefill": W.prefill}[workload]
            self.wl = make() if seed is None else make(seed=seed)
        self.wl.kv_format = kv_format
        self.workload = workload
        self.dw = DeviceWorkload(self.wl, device=device)
        wl, dw = self.wl, self.dw
        # T new tokens per sequence (the step's queries: 1 for decode, Q for a
        # multi-token step, the chunk for prefill), T / m new entries
        B, T, m = wl.batch, wl.nq, wl.m
        Q = T
        self.queries = T
        # several new tokens: their window rows are written by the FP8 quantiser
        # right before each layer call, so keys may not be read ahead of it
        dw.early_inputs = T == 1
        # one new token: every layer's q and window row are in place before the
        # step, so a Reuse layer's whole attention may run ahead of its dependency
        # wait (csa2.ATTN_EARLY_ALL; Reuse layers alternate between two workspaces)
        dw.early_all = T == 1 and early_all
        dev = dw.dev
        Ns = [wl.tokens[b] for b in range(B)]
        N = Ns[0]
        self.new_slots = torch.cat([dw.entry_slots(b, (Ns[b] - T) // m, Ns[b] // m) for b in range(B)])
        self.C_new = torch.cat([synth.normal_bf16_torch(wl._sid(W.T_C, b), (Ns[b] - T) * 512, T * 512, dev)
                                for b in range(B)]).view(B * T, 512)
        self.Z_new = torch.cat([synth.normal_bf16_torch(wl._sid(W.T_Z, b), (Ns[b] - T) * 512, T * 512, dev)
                                for b in range(B)]).view(B * T, 512) if m > 1 else torch.zeros_like(self.C_new)
        self.bias = torch.from_numpy(wl.bias()).to(dev) if m > 1 else \
            torch.zeros((1, 512), dtype=torch.float32, device=dev)
        self.ik_new = torch.cat([synth.normal_f32_torch(wl._sid(W.T_IK, b), (Ns[b] - T) // m * 128, T // m * 128, dev)
                                 for b in range(B)]).view(B * T // m, 128)
        self.swa_new = {l: torch.cat([synth.normal_bf16_torch(wl._sid(W.T_SWA, b, l), (Ns[b] - T) * 512, T * 512, dev)
                                      for b in range(B)]).view(B * T, 512).float() for l in dw.layers}
        R = wl.swa_rows
        self.ring_slots = torch.tensor([b * R + (Ns[b] - T + i) % R for b in range(B) for i in range(T)],
                                       dtype=torch.int64, device=dev)
        self.scan_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in self.scan_ev:
            e.record()                       # materialise the CUDA events
        self.set_schedule()
        # the step's host-fed inputs (new tokens, every layer's queries and window
        # rows) in two device buffers -- the first IN_EARLY layers' / the rest --
        # and its outputs (every layer's o and lse) in one buffer per group of
        # OUT_GROUP layers, so that the end-to-end leg copies the later layers'
        # inputs in once the first layer's HBM-bound scan is over (a copy beside
        # the scan slows it by about the copy's own time) while the next layers
        # run, and each group's outputs out while the later layers run
        layers = list(dw.layers)
        early, _, self.out_groups = e2e_groups(len(layers))
        ins0 = [(self.__dict__, "C_new"), (self.__dict__, "ik_new")]
        ins1 = []
        for i, l in enumerate(layers):
            refs = [(dw.q, l), (self.swa_new, l)] + ([(dw.qi, l), (dw.w, l)] if l in dw.qi else [])
            (ins0 if i in early else ins1).extend(refs)
        self.in_dev = [self._gather(ins0)] + ([self._gather(ins1)] if ins1 else [])
        outs = [[(dw.o, l), (dw.lse, l)] for l in layers]
        self.out_dev = [self._gather(sum([outs[i] for i in g], [])) for g in self.out_groups]

    def set_schedule(self):
        """The attention schedule the library takes for this step, and the step's
        kernel launches: Full (scan, block Top-2,048, pool Top-512) and Reindex
        (rescoring, select) ahead of the attention, which is one launch in the
        row schedule and two (attention, merge) in the chunk schedule; the new
        entries' launch; with several new tokens, their window rows per layer."""
        csa2, dw, wl = self.csa2, self.dw, self.wl
        l0 = dw.layers[0]
        self.schedule = csa2.csa2_sparse_attn_schedule(
            dw.batch, dw.swa(l0, new_rows=self.swa_new[l0] if self.queries == 1 else None))
        attn = 1 if self.schedule == csa2.ATTN_SCHEDULE_ROWS else 2
        self.launches = 1 + sum({"full": 3, "reindex": 2, "reuse": 0}[m] + attn for m in wl.layers) + \
            (len(wl.layers) if self.queries > 1 else 0)

    def _gather(self, refs):
        """One device byte buffer holding the tensors refs name (container, key),
        each 256-byte aligned; the containers are rebound to views of it."""
        torch = self.torch
        sizes = [(c[k].numel() * c[k].element_size() + 255) // 256 * 256 for c, k in refs]
        buf = torch.empty(sum(sizes), dtype=torch.uint8, device=self.dw.dev)
        off = 0
        for (c, k), n in zip(refs, sizes):
            t = c[k]
            v = buf[off: off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            c[k] = v
            off += n
        return buf

    def enqueue(self, prof=True):
        csa2, dw, cache = self.csa2, self.dw, self.dw.cache
        # the new token's entry (m = 1): compressed, its FP4 main KV and FP8 indexer key into the cache
        csa2.csa2_append_entries(self.dw.cstruct, self.C_new, self.Z_new, self.bias, self.wl.m, self.ik_new,
                                 slots=self.new_slots)
        self.enqueue_layers(dw.layers, prof)

    def enqueue_e2e(self, host_in, host_out, s2, s3):
        """The step with its copies, for capture on the current stream: the first
        IN_EARLY layers' inputs first; the other layers' on s2 once the first
        layer has run, while the next ones run; each group of layers' outputs on
        s3 once its last layer has run, the last group's at the end."""
        torch, dw, csa2 = self.torch, self.dw, self.csa2
        s = torch.cuda.current_stream()
        ev_in = torch.cuda.Event()
        ev_out = [torch.cuda.Event() for _ in self.out_groups]
        self.in_dev[0].copy_(host_in[0], non_blocking=True)
        csa2.csa2_append_entries(self.dw.cstruct, self.C_new, self.Z_new, self.bias, self.wl.m, self.ik_new,
                                 slots=self.new_slots)
        layers = list(dw.layers)
        last = {g[-1]: gi for gi, g in enumerate(self.out_groups)}
        for i, l in enumerate(layers):
            if i == IN_EARLY:
                s.wait_event(ev_in)
            self.enqueue_layers([l])
            if i == 0 and len(self.in_dev) > 1:
                s2.wait_stream(s)
                with torch.cuda.stream(s2):
                    self.in_dev[1].copy_(host_in[1], non_blocking=True)
                    ev_in.record(s2)
            gi = last.get(i)
            if gi is not None and gi < len(self.out_groups) - 1:
                ev_out[gi].record(s)
                s3.wait_event(ev_out[gi])
                with torch.cuda.stream(s3):
                    host_out[gi].copy_(self.out_dev[gi], non_blocking=True)
        host_out[-1].copy_(self.out_dev[-1], non_blocking=True)
        if len(self.in_dev) > 1:
            s.wait_stream(s2)
        if len(self.out_dev) > 1:
            s.wait_stream(s3)

    def enqueue_layers(self, layers, prof=False):
        for l in layers:
            # the layer; its attention call also quantises this layer's window
            # row of the new token into the ring (csa2_swa.new_rows); several new
            # tokens per sequence: the FP8 quantiser writes their rows first
            full = self.wl.layers[l] == "full"
            if self.queries > 1:
                dw = self.dw
                self.csa2.csa2_quant_fp8(self.swa_new[l], dw.swa_codes[l].view(-1, 512), dw.swa_scales[l].view(-1),
                                         slots=self.ring_slots, status=dw.cache.status)
            self.dw.run_layer(l, prof=self.scan_ev if (prof and full) else None,
                              new_rows=self.swa_new[l] if self.queries == 1 else None)

    def rows_visible(self):
        return rows_visible(self.wl)

    def layer_bytes(self):
        return layer_bytes(self.wl)

    def scan_work(self):
        return scan_work(self.wl)


# ---------------------------------------------------------------- algorithmic work
KV_SCALE_BYTES = {0: 16, 1: 32}     # main-KV block-scale bytes per entry: MXFP4, FP4 with E4M3 per 16
OUT_GROUP = 2                       # e2e: layers whose outputs go back to the host in one copy
IN_EARLY = 5                        # e2e: layers whose inputs are copied in before the step's kernels


def e2e_groups(n_layers):
    """The end-to-end leg's copies by layer position: the layers whose inputs
    go in before the step's kernels, those whose inputs go in once the first
    layer has run, and the groups of layers whose outputs go out together
    (pairs, the last layer alone: the copy after the last kernel is short)."""
    early = list(range(min(IN_EARLY, n_layers)))
    late = list(range(len(early), n_layers))
    out = [list(range(g, min(g + OUT_GROUP, n_layers))) for g in range(0, n_layers, OUT_GROUP)]
    if out and len(out[-1]) > 1:
        out[-1:] = [out[-1][:-1], out[-1][-1:]]
    return early, late, out
POOL_MAX = 16384                    # candidate pool: 2,048 blocks of 8


def rows_visible(wl):
    """Entries visible to each query row of the step (causal, m tokens per entry)."""
    out = []
    for b in range(wl.batch):
        E = wl.entries(b)
        out += [min(E, (int(t) + 1) // wl.m) for t in wl.q_pos(b)]
    return out


def layer_bytes(wl):
    """Algorithmic bytes per step of each layer mode, all sequences: what the
    method must read and write -- the indexer keys scanned (once for all of a
    sequence's query tokens) or rescored, and per query token the selected
    main-KV entries, the window rows, q / qi / w, the pool or indices, o and
    lse."""
    kv = 256 + KV_SCALE_BYTES[wl.kv_format]                  # codes + block scales per entry
    attn = 512 * kv + 128 * 516 + 64 * 512 * 2 + 64 * 512 * 4 + 64 * 4
    vis = rows_visible(wl)
    keys = sum(wl.entries(b) for b in range(wl.batch)) * 132
    full = keys + sum((v // 8) * 4 + 32 * 128 * 2 + 32 * 4 + attn for v in vis)
    reindex = sum(min(POOL_MAX, v) * 136 + 32 * 128 * 2 + 32 * 4 + attn for v in vis)
    reuse = len(vis) * (512 * 4 + attn)
    return {"full": full, "reindex": reindex, "reuse": reuse}


def scan_work(wl):
    """The Full layer scan's algorithmic work per launch: HBM bytes (keys once
    per sequence, block maxima, queries) or, for a prefill chunk, where the
    keys stay in L2 and the products bound it, e4m3 FLOPs."""
    vis = rows_visible(wl)
    if wl.nq > 4:
        return "tensor", sum(vis) * 32 * 128 * 2.0
    return "hbm", float(sum(wl.entries(b) for b in range(wl.batch)) * 132 +
                        sum((v // 8) * 4 + 8192 + 128 for v in vis))


def run_native(args):
    import torch
    import torch.distributed as dist
    from compressed_sparse_attention_layer_gb300 import build, csa2

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    build.build()
    csa2.load()
    dev = torch.device("cuda", local)
    seed = rank_seed(rank) if args.workload == "decode_1m" else None
    step = DecodeStep(args.batch, args.tokens, seed, dev, kv_format=args.kv_format, queries=args.queries,
                      workload=args.workload, early_all=not args.no_early_all)
    B, N, Q = step.wl.batch, step.wl.tokens[0], step.queries
    if args.bf16_scores:
        step.dw.layer_flags |= csa2.LAYER_SCORES_BF16
    if args.e4m3_query:
        step.dw.layer_flags |= csa2.LAYER_INDEX_E4M3_QUERY
    if args.attn_schedule != "auto":
        sch = {"chunks": csa2.ATTN_SCHEDULE_CHUNKS, "rows": csa2.ATTN_SCHEDULE_ROWS}[args.attn_schedule]
        step.dw.attn_options["flags"] = step.dw.attn_options.get("flags", 0) | sch
        step.set_schedule()

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.enqueue()                                   # eager warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.enqueue()
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()

    # ---- timed region (device-resident inputs)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    scan_ms = []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.nvtx.range_push("csa2_timed")
    flush = None
    if sum(step.wl.entries(b) for b in range(B)) * 132 < (256 << 20):
        # the step's indexer keys fit in L2: flush it before every timed step
        # (a 512 MB write) and time each step alone
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    ms = 0.0
    with torch.cuda.stream(s):
        if flush is None:
            ev0.record(s)
            for _ in range(args.steps):
                g.replay()
            ev1.record(s)
    if flush is not None:
        for _ in range(args.steps):
            with torch.cuda.stream(s):
                flush.fill_(1)
                ev0.record(s)
                g.replay()
                ev1.record(s)
            torch.cuda.synchronize()
            ms += ev0.elapsed_time(ev1)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    if flush is None:
        ms = ev0.elapsed_time(ev1)
    # dominant-kernel duration: the scan events recorded inside the graph, once per replay
    for _ in range(min(args.steps, 10)):
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        scan_ms.append(step.scan_ev[0].elapsed_time(step.scan_ev[1]))
    # per layer mode: the step's layers of one mode captured back to back in a
    # graph of their own (the same launches, the same programmatic overlap
    # between consecutive layers), replayed after the timed region
    per_mode_ms = {}
    for mode in ("full", "reindex", "reuse"):
        ls = [l for l in step.dw.layers if step.wl.layers[l] == mode]
        if not ls:
            continue
        reps = max(1, 8 // len(ls))
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm, stream=s):
            for _ in range(reps):
                step.enqueue_layers(ls)
        torch.cuda.synchronize()
        t = []
        for _ in range(5):
            with torch.cuda.stream(s):
                ev0.record(s)
                gm.replay()
                ev1.record(s)
            torch.cuda.synchronize()
            t.append(ev0.elapsed_time(ev1) / (reps * len(ls)))
        per_mode_ms[mode] = (len(ls), statistics.median(t))
        del gm
    ms_total = reduce_max(ms, dev, world)
    ms_step = ms_total / args.steps
    value = throughput(world, B * Q, args.steps, ms_total / 1e3)

    # ---- end to end: pinned host inputs copied in, outputs copied out, every step
    # (one graph per step with its copies; within a step the copies overlap the
    # layers that do not need them)
    e2e = None
    if not args.no_e2e:
        host_in = [x.cpu().pin_memory() for x in step.in_dev]
        host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in step.out_dev]
        h2d_bytes = sum(h.numel() * h.element_size() for h in host_in)
        d2h_bytes = sum(h.numel() * h.element_size() for h in host_out)
        s2, s3 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=s):
            step.enqueue_e2e(host_in, host_out, s2, s3)
        torch.cuda.synchronize()
        for _ in range(2):
            with torch.cuda.stream(s):
                ge.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            with torch.cuda.stream(s):
                ge.replay()
            s.synchronize()
        el = time.perf_counter() - t0
        e2e = {"value": throughput(world, B * Q, args.steps, reduce_max(el, dev, world)), "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes}
        del ge

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel (the Full layer's index scan)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    bound, work = step.scan_work()
    scan_avg = statistics.median(scan_ms) if scan_ms else None
    if bound == "hbm":
        achieved = work / (scan_avg * 1e-3) / 1e9 if scan_avg else None
        unit_r = "GB/s"
    else:
        # e4m3 products: the measured bf16 sustained peak x 2 (the nominal fp8 / bf16 ratio)
        peak = 2.0 * peaks.get("bf16_tflops_sustained", 1700.0)
        achieved = work / (scan_avg * 1e-3) / 1e12 if scan_avg else None
        unit_r = "TFLOP/s"
    traffic = None
    prof_path = os.path.join(ROOT, "profiles", "traffic_index_scan.json")
    if os.path.exists(prof_path):
        try:
            with open(prof_path) as f:
                tp = json.load(f)
            if tp.get("kernel_version") == KERNEL_VERSION:
                traffic = tp.get("bytes_per_launch")
        except (OSError, ValueError):
            pass
    if args.workload != "decode_1m" or Q != 1 or N != 1 << 20 or B != 8:
        traffic = None                     # the ncu record is of the headline workload's launch
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit_r,
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "kernel": "index scan (Full layer)", "kernel_ms": scan_avg,
                "peak_source": ("MEASURED_PEAKS.json hbm_gbs (measured)" if "hbm_gbs" in peaks else "fallback")
                if bound == "hbm" else "MEASURED_PEAKS.json bf16_tflops_sustained x 2 (e4m3 / bf16 nominal ratio)"}
    hbm_peak = peaks.get("hbm_gbs", 6800.0)

    # per layer mode: median layer time, query tokens/s of that layer alone, and its
    # algorithmic bytes over that time against the same peak
    lb = step.layer_bytes()
    per_mode = {}
    rows = B * Q
    for mode, (n, lms) in per_mode_ms.items():
        gbs = lb[mode] / (lms * 1e-3) / 1e9
        per_mode[mode] = {"layers": n, "us_per_layer": 1e3 * lms, "query_tokens_per_s": rows / (lms * 1e-3),
                          "algo_bytes_per_token": lb[mode] / rows, "achieved_gbs": gbs, "frac": gbs / hbm_peak}
    stack_bytes = sum(lb[m] for m in step.wl.layers)
    rest = ms_step - sum(n * lms for n, lms in per_mode_ms.values())
    per_mode["stack"] = {"us": 1e3 * ms_step, "algo_bytes_per_token": stack_bytes / rows,
                         "achieved_gbs": stack_bytes / (ms_step * 1e-3) / 1e9,
                         "frac": stack_bytes / (ms_step * 1e-3) / 1e9 / hbm_peak,
                         "us_outside_layers": 1e3 * rest,
                         "note": "layer times: each mode's layers of the step captured back to back in a "
                                 "graph of their own; outside: the new token's quantisation and launch gaps"}
    # the whole step against the same HBM peak: algorithmic bytes of every layer over the step time
    roofline["step_frac"] = per_mode["stack"]["frac"]
    roofline["step_achieved_gbs"] = per_mode["stack"]["achieved_gbs"]

    cpu = None
    if not args.no_cpu_baseline and step.wl.nq == 1:
        cpu = cpu_baseline(step.wl)
    wl = step.wl
    if args.workload == "decode_1m":
        wdesc = (f"decode_1m: batch {B} x {N} tokens" if Q == 1 else
                 f"decode_multi: batch {B} x {N} tokens, {Q} query tokens per sequence per step") + \
            ", m=1, 20-layer decoder stack (Full+3 Reuse, 4x(Reindex+3 Reuse)), Top-512, SWA 128"
    elif args.workload == "prefill":
        wdesc = (f"prefill: one chunk of {wl.nq} new tokens after {N - wl.nq}, m={wl.m} "
                 f"({wl.entries(0)} entries), causal, Full + 5 Reuse, Top-512, SWA 128")
    else:
        lens = [wl.tokens[b] for b in range(B)]
        wdesc = (f"{args.workload}: batch {B}, contexts {min(lens)}..{max(lens)} tokens (mean {sum(lens) // B}), "
                 f"m={wl.m}, {len(wl.layers)} layers {'/'.join(sorted(set(wl.layers)))}, Top-512, SWA 128")
    inputs_bytes = sum(wl.entries(b) for b in range(B)) * 132

    metric = METRIC if args.workload == "decode_1m" and Q == 1 and not args.bf16_scores and not args.e4m3_query \
        else f"CSA2 query-tokens/s, {args.workload}" + (f", {Q} query tokens per sequence" if Q > 1 else "") + \
        (", bf16 index scores" if args.bf16_scores else "") + (", one-part e4m3 index query" if args.e4m3_query else "")
    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3/bf16",
        "data": "synthetic (seeded counter-based generator; 64 planted blocks per sequence)",
        "config": {"workload": wdesc,
                   "queries_per_sequence": Q,
                   "batch": B, "context_tokens": N, "layers": len(step.wl.layers),
                   "main_kv": ["MXFP4 (32-element blocks, E8M0 scale), 272 B/entry",
                               "FP4 (16-element blocks, E4M3 scale), 288 B/entry"][args.kv_format],
                   "l2": (f"inputs larger than L2: the Full layer scans {inputs_bytes / 1e9:.2f} GB of indexer "
                          "keys per step") if inputs_bytes >= (256 << 20) else
                         (f"L2 flushed (512 MB write) before every timed step; the step's indexer keys are "
                          f"{inputs_bytes / 1e6:.1f} MB"),
                   "graph": "one CUDA graph per step",
                   "index_scores": "bf16 (selection on rounded scores)" if args.bf16_scores else "fp32",
                   "index_query": "one e4m3 part per head" if args.e4m3_query else "two e4m3 parts (hi + lo)",
                   "attention": "persistent clusters over whole rows" if step.schedule == csa2.ATTN_SCHEDULE_ROWS
                   else "one cluster per (row, 128-key chunk) and a merge"},
        "roofline": roofline, "per_layer_mode": per_mode, "clocks": clk, "e2e": e2e, "gpu_launches": step.launches * args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


KERNEL_VERSION = "f8-cpasync-scan-v6"
NORM_ROPE_VERSION = "norm-rope-int-turns-v1"   # the prologue kernel whose ncu traffic profiles/ records


# ---------------------------------------------------------------- CPU oracle
_SAMPLES = {}


def _prepare(wl, b):
    """Oracle-side inputs of sequence b (its cache, window rings, queries): not timed."""
    from tests.reference import SeqOracle
    key = (wl.name, wl.seed, b)
    if key not in _SAMPLES:
        so = SeqOracle(wl, b)
        so.ik()
        rings = {l: so.swa_ring(l) for l in range(len(wl.layers))}
        qs = {l: (wl.qi_bits(l, b, [0])[0], wl.w(l, b, [0])[0], wl.q_bits(l, b, [0])[0])
              for l in range(len(wl.layers))}
        _SAMPLES[key] = (so, rings, qs)
    return _SAMPLES[key]


def oracle_sample(wl, b=0, layers=None):
    """Run the oracle through the decoder layers for sequence b's decode token.
    Returns seconds spent in the oracle (inputs generated beforehand)."""
    import numpy as np
    import oracle

    so, rings, qs = _prepare(wl, b)
    t0 = time.perf_counter()
    idx = pool = None
    codes, scales = so.ik()
    _, nvis = so.visible(0)
    t = int(wl.q_pos(b)[0])
    for l, mode in enumerate(wl.layers[:layers]):
        qi, w, q = qs[l]
        if mode == "full":
            idx, pool, _ = oracle.full_select(qi, w, codes, scales, nvis)
        elif mode == "reindex":
            idx, _ = oracle.reindex_select(qi, w, codes, scales, pool)
        sel = idx[idx >= 0]
        kvc, kvs = so.kv(sel)
        keys = oracle.attention_keys(kvc, kvs, np.arange(sel.size, dtype=np.int32), rings[l][0], rings[l][1], t)
        oracle.attention(q, 1.0, keys)
    return time.perf_counter() - t0


def cpu_baseline(wl, target_s=10.0):
    """The oracle on the host cores over one decode step's query tokens (every
    sequence's token through all layers), each repeated so the timed oracle
    work comes to about target_s seconds; inputs are prepared outside the timing."""
    import math
    import oracle
    secs, n, reps = 0.0, 0, None
    seqs = range(0, wl.batch, max(1, wl.batch // 8))            # at most 8 sequences, spread over the batch
    for b in seqs:
        s0 = oracle_sample(wl, b)
        if reps is None:
            reps = max(1, math.ceil(target_s / (s0 * len(seqs))))
        secs += s0 + sum(oracle_sample(wl, b) for _ in range(reps - 1))
        n += reps
        _SAMPLES.pop((wl.name, wl.seed, b), None)
    nb = len(seqs)
    return {"value": n / secs, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the decode query tokens of {nb} of the step's {wl.batch} sequences, each {reps}x, "
                      f"through all {len(wl.layers)} layers at their contexts ({wl.tokens[0]} tokens for the "
                      f"first); {n} tokens in {secs:.1f} s of oracle time"}


def run_norm_rope(args):
    """The attention inputs' prologue (csa2_norm_rope) on a prefill chunk's
    queries: 8,192 tokens x 64 heads of 512 fp32 dims, RMS-normalised and
    rotated at their positions, written as bf16.  HBM bound: 2,048 B read and
    1,024 B written per vector (1.61 GB per launch, above L2)."""
    import torch
    from compressed_sparse_attention_layer_gb300 import build, csa2, synth
    world, rank, local = dist_env()
    if rank != 0:
        return                                  # one GPU: the prologue does not shard across ranks here
    torch.cuda.set_device(local)
    build.build()
    csa2.load()
    dev = torch.device("cuda", local)
    T, H = 8192, 64
    x = synth.normal_f32_torch(7100, 0, T * H * 512, dev).view(T, H, 512)
    gamma = (1.0 + 0.1 * synth.normal_f32_torch(7101, 0, 512, dev)).contiguous()
    pos = torch.arange(65536, 65536 + T, dtype=torch.int64, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)

    def launch():
        csa2.csa2_norm_rope(x, out, gamma, 1e-6, pos, 10000.0, stream=s)

    with torch.cuda.stream(s):
        for _ in range(max(3, args.warmup)):
            launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    e0.record(s)
    for _ in range(args.steps):
        launch()
    e1.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    nvec = T * H
    # end to end: pinned host input copied in, the prologue, bf16 result copied out
    hx = torch.empty((T, H, 512), dtype=torch.float32, pin_memory=True)
    hx.copy_(x)
    ho = torch.empty((T, H, 512), dtype=torch.bfloat16, pin_memory=True)
    torch.cuda.synchronize()
    def e2e_step():
        with torch.cuda.stream(s):
            x.copy_(hx, non_blocking=True)
            launch()
            ho.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    s.synchronize()
    e2e_s = (time.perf_counter() - t0) / max(1, args.steps)
    algo = nvec * (2048 + 1024)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    achieved = algo / (ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_norm_rope.json")) as f:
            tp = json.load(f)
        if tp.get("kernel_version") == NORM_ROPE_VERSION:
            traffic = tp["bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    line = {"metric": "CSA2 input prologue (RMSNorm + partial RoPE) vectors/s, 8,192 tokens x 64 heads",
            "value": nvec / (ms * 1e-3), "unit": "vectors/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": "norm_rope: 8,192 query tokens x 64 heads x 512 dims, fp32 in, bf16 out, "
                                   "positions 65,536.., rope_base 10,000",
                       "l2": "inputs larger than L2 (1.07 GB read per launch)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "kernel": "k_norm_rope",
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if "hbm_gbs" in peaks
                         else "fallback"},
            "clocks": clk,
            "e2e": {"value": nvec / e2e_s, "unit": "vectors/s", "h2d_bytes_per_step": hx.numel() * 4,
                    "d2h_bytes_per_step": ho.numel() * 2},
            "gpu_launches": args.steps, "cpu_baseline": None}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = norm_rope_cpu_baseline()
    print(json.dumps(line))


def norm_rope_cpu_baseline(reps=20):
    """The oracle's RMSNorm + RoPE on the host: 256 of the chunk's tokens x 64
    heads, repeated reps times (about 1.5 s), inputs prepared outside the timing."""
    import numpy as np
    import oracle
    from compressed_sparse_attention_layer_gb300 import synth
    oracle.build()
    T, H = 256, 64
    x = synth.normal_f32(7100, 0, T * H * 512).reshape(T, H, 512)
    gamma = (1.0 + 0.1 * synth.normal_f32(7101, 0, 512)).astype(np.float32)
    pos = np.arange(65536, 65536 + T, dtype=np.int64)
    oracle.norm_rope(x, gamma, 1e-6, pos, 10000.0)          # warm-up (library load)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.norm_rope(x, gamma, 1e-6, pos, 10000.0)
    secs = time.perf_counter() - t0
    return {"value": reps * T * H / secs, "unit": "vectors/s", "cores": 1, "kind": "oracle",
            "sample": f"{T} of the 8,192 query tokens x {H} heads, {reps}x ({reps * T * H} vectors in "
                      f"{secs:.1f} s, single-threaded)"}


def run_reference_norm_rope(args):
    """The oracle's RMSNorm + RoPE on a bounded sample of the prologue
    workload: each step 256 of the chunk's 8,192 query tokens (x 64 heads)."""
    import numpy as np
    import oracle
    from compressed_sparse_attention_layer_gb300 import synth
    oracle.build()
    T, H = 256, 64
    x = synth.normal_f32(7100, 0, T * H * 512).reshape(T, H, 512)
    gamma = (1.0 + 0.1 * synth.normal_f32(7101, 0, 512)).astype(np.float32)
    pos = np.arange(65536, 65536 + T, dtype=np.int64)
    for _ in range(max(1, min(args.warmup, 1))):
        oracle.norm_rope(x, gamma, 1e-6, pos, 10000.0)
    tot = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.norm_rope(x, gamma, 1e-6, pos, 10000.0)
        tot += time.perf_counter() - t0
    value = args.steps * T * H / tot
    sample = f"each step: {T} of the 8,192 query tokens x {H} heads ({T * H} vectors), single-threaded oracle"
    print(json.dumps({"impl": "reference", "metric": "CSA2 input prologue (RMSNorm + partial RoPE) vectors/s, "
                      "8,192 tokens x 64 heads", "value": value, "unit": "vectors/s", "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic", "config": {"workload": "norm_rope: 8,192 query tokens x 64 heads x "
                                                                  "512 dims (sampled)"},
                      "cpu_baseline": {"value": value, "unit": "vectors/s", "cores": 1, "kind": "oracle",
                                       "sample": sample},
                      "e2e": {"value": value, "unit": "vectors/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    if args.workload == "norm_rope":
        return run_reference_norm_rope(args)
    import oracle
    from compressed_sparse_attention_layer_gb300 import workloads as W
    oracle.build()
    wl = W.decode_1m(seed=4000, batch=args.batch, tokens=args.tokens)
    for _ in range(args.warmup and 1):
        oracle_sample(wl, 0, layers=1)
    tot = 0.0
    for k in range(args.steps):
        tot += oracle_sample(wl, 0)
    value = args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"decode_1m: batch {wl.batch} x {wl.tokens[0]} tokens"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"each step: 1 decode query token of one sequence through "
                                       f"{len(wl.layers)} layers"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.workload == "norm_rope":
        run_norm_rope(a)
    else:
        run_native(a)
