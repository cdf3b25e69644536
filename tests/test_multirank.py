"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The decode batch partitions: every rank runs its own sequences and the only
cross-rank traffic is the barrier and the maximum of the elapsed times.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from compressed_sparse_attention_layer_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = [12.5, 20.0][rank]                 # the second rank is slower
        ms = bench.reduce_max(local_ms, "cpu", world)
        out[rank] = (ms, bench.throughput(world, 8, 10, ms / 1e3))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 20.0
    assert value == pytest.approx(2 * 8 * 10 / 0.020)


def test_ranks_decode_different_sequences():
    """Weak scaling: rank r's batch comes from its own seed, so the shards differ."""
    a = W.decode_1m(seed=bench.rank_seed(0), batch=2, tokens=4096)
    b = W.decode_1m(seed=bench.rank_seed(1), batch=2, tokens=4096)
    assert bench.rank_seed(0) != bench.rank_seed(1)
    assert not (a.q_bits(0, 0, [0]) == b.q_bits(0, 0, [0])).all()


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.0, "cpu", 1) == 3.0
    assert bench.throughput(1, 8, 20, 0.5) == 320.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, batch, tokens = 1, 1, 8, 1 << 20

    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""
