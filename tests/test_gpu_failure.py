"""The bounded device waits, driven to run out on purpose (needs a GPU).

Every wait of the tensor-core kernels -- the index scan's pipeline barriers
and the attention's product commits -- gives up after a bounded number of
polls, sets CSA2_DEV_TIMEOUT in the cache's status word and lets the kernel
finish normally.  csa2_debug_set_wait_limit(1) leaves each of those waits a
single poll, which a wait issued right after its copies or products cannot
meet: the layer calls return, the status word carries the timeout, and a
normal call on the same context afterwards is at parity with the oracle.
Nothing here faults or hangs the GPU: the waits end by themselves and the
kernels' in-flight copies and products are awaited (long limit) before their
shared and tensor memory are released.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_layer_gb300 import csa2
from compressed_sparse_attention_layer_gb300 import workloads as W
from compressed_sparse_attention_layer_gb300.device import DeviceWorkload
from tests.test_gpu_layers import _check_sequence, _run_recording

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from compressed_sparse_attention_layer_gb300 import build
    build.build()
    csa2.load()


def test_waits_time_out_and_the_context_stays_usable():
    wl = W.Workload("timeout", 81, 2, [5000, 30000], 1, ["full", "reuse", "reindex"], planted_blocks=2)
    dw = DeviceWorkload(wl)
    csa2.csa2_debug_set_wait_limit(1)
    try:
        for l in dw.layers:
            dw.run_layer(l, new_rows=dw.swa_new_rows(l))
        torch.cuda.synchronize()                      # every call returned and its kernels finished
    finally:
        csa2.csa2_debug_set_wait_limit(0)
    status = int(dw.cache.status[0])
    assert status & csa2.DEV_TIMEOUT, status
    # no page or slot went out of range (the selection that followed an aborted
    # scan ranked undefined scores, but only ever of visible entries)
    assert not (status & (csa2.DEV_BAD_PAGE | csa2.DEV_BAD_SLOT)), status
    # the same context, the default limit: the layers are at parity again
    fresh = DeviceWorkload(wl)
    _run_recording(fresh)
    for b in range(wl.batch):
        _check_sequence(fresh, b)
    assert int(fresh.cache.status[0]) == 0


def test_row_schedule_waits_time_out_and_the_context_stays_usable():
    """The persistent row schedule of the attention under a one-poll limit:
    every wait of its item loop runs out first (flagged), then waits for the
    same phase once more with the long limit, so the two CTAs of a cluster
    keep the same sequence of exchanges and the call completes."""
    wl = W.Workload("timeout_rows", 82, 2, [5000, 30000], 1, ["full", "reuse"], planted_blocks=2,
                    nq=3, prefill_new=3, swa_rows=W.W + 3)
    dw = DeviceWorkload(wl)
    dw.attn_options = dict(flags=csa2.ATTN_SCHEDULE_ROWS)
    csa2.csa2_debug_set_wait_limit(1)
    try:
        for l in dw.layers:
            dw.run_layer(l)
        torch.cuda.synchronize()
    finally:
        csa2.csa2_debug_set_wait_limit(0)
    status = int(dw.cache.status[0])
    assert status & csa2.DEV_TIMEOUT, status
    assert not (status & (csa2.DEV_BAD_PAGE | csa2.DEV_BAD_SLOT)), status
    fresh = DeviceWorkload(wl)
    fresh.attn_options = dict(flags=csa2.ATTN_SCHEDULE_ROWS)
    _run_recording(fresh)
    for b in range(wl.batch):
        for i in range(wl.nq):
            _check_sequence(fresh, b, i)
    assert int(fresh.cache.status[0]) == 0
