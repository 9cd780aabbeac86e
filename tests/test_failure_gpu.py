"""The failure path on the GPU without a fault: a short wait limit and one
withheld loader-to-MMA hand-off make a pipeline wait run out. The call must
come back with SMQ_ERR_TIMEOUT in the status word (the kernel winds down:
bounded waits for its own copies, drained MMAs, TMEM freed), and the next
normal call on a re-initialised workspace must match the oracle. Every wait
stays bounded; nothing faults, traps or hangs."""

import time

import numpy as np
import pytest

import oracle
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import synth, tensors

from gpu_check import check_rows

pytestmark = pytest.mark.gpu

SHORT_NS = 2_000_000  # 2 ms


def _stall_then_recover(inp, run, make):
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    dev = make(inp, plan)
    plan.set_wait_limit(SHORT_NS)
    plan.inject_stall(1)
    t0 = time.perf_counter()
    run(dev, plan)
    status = smq.smq_get_status(dev.workspace)
    elapsed = time.perf_counter() - t0
    assert status & smq.SMQ_ERR_TIMEOUT, f"status {status}: the withheld hand-off must time out"
    assert elapsed < 5.0, f"the stalled call took {elapsed:.2f} s"
    plan.inject_stall(-1)
    plan.set_wait_limit(2_000_000_000)
    smq.smq_workspace_init(plan, dev.workspace)
    run(dev, plan)
    assert smq.smq_get_status(dev.workspace) == 0
    return plan, dev


def _decode(dev, plan):
    dev.run(plan)


def _prefill(dev, plan):
    dev.gather(plan)
    dev.run(plan)


def test_timeout_in_the_row_cluster_kernel():
    inp = synth.decode_batch(seed=91, rows=16)
    plan, dev = _stall_then_recover(inp, _decode, tensors.DecodeDevice)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, rows=range(0, 16, 3), mode="sparse"))


def test_timeout_in_the_persistent_kernel():
    inp = synth.multi_token_decode(seed=93, requests=80, next_n=2, ctx_range=(1000, 5000), ncb=16, topk=300)
    assert inp.rows > 152  # more rows than SMs: the persistent score kernel and the top-k kernel
    plan, dev = _stall_then_recover(inp, _decode, tensors.DecodeDevice)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, rows=range(0, inp.rows, 11), mode="sparse"))


def test_timeout_in_the_tensor_copy_paths():
    pf = synth.prefill_chunk(seed=95, seq_lens=(1500, 2300), queries_per_seq=90, num_heads=64, page_size=64,
                             cbs=128, ncb=8, topk=200)
    kv, ks = oracle.gather_reference(pf)
    for window_major in (True, False):  # the window-major kernel; the row-major one on the contiguous workspace
        plan, dev = _stall_then_recover(pf, _prefill,
                                        lambda i, p, wm=window_major: tensors.PrefillDevice(i, p, window_major=wm))
        check_rows(pf, dev, plan,
                   oracle.reference_rows(pf, rows=range(0, pf.rows, 13), mode="sparse", contig=(kv, ks)))
    dec = synth.prefill_as_decode(pf)  # 180 rows on 2 block-table rows: paged tensor copies
    plan, dev = _stall_then_recover(dec, _decode, tensors.DecodeDevice)
    check_rows(dec, dev, plan, oracle.reference_rows(dec, rows=range(0, dec.rows, 13), mode="sparse"))
