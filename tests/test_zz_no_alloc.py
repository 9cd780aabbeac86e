"""The scratch-free decode entry point against the workspace one.

sparse_mqa_logits_topk_decode_noalloc runs the same kernels on the library's
static device scratch instead of a caller's workspace.  Both entry points are
called through the C ABI on the same inputs, twice in a row with different
shapes, and must give the same bytes.  This file is collected last so that it
also runs after every other GPU test in one process.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import synth, tensors

from oracle import check
from gpu_check import check_rows

pytestmark = pytest.mark.gpu


def _outputs(dev):
    return dev.topk_out.clone(), dev.col_indices.clone(), dev.sparse_indices.clone(), dev.end.clone()


def _run_noalloc(plan, dev):
    smq.sparse_mqa_logits_topk_decode_noalloc(plan, dev.q, dev.q_scale, dev.weights, dev.k_cache, dev.block_table,
                                              dev.row_indices, dev.row_ke, dev.candidate_blocks, dev.topk_out,
                                              dev.sparse_indices, dev.end, col_indices=dev.col_indices)


def _check_oracle(inp, dev, plan, ref):
    """Structure of every row, and the top-k sets of the oracle's rows (the
    logits stay in the library's scratch)."""
    check_rows(inp, dev, plan, {})
    top = tensors.to_numpy(dev.topk_out)
    for r, row in ref.items():
        check.check_topk(top[r], row, inp.geom.topk, f"row {r} top-k")


def _compare(inp):
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    with_ws = tensors.DecodeDevice(inp, plan, with_logits=False)
    with_ws.run(plan)
    assert smq.smq_get_status(with_ws.workspace) == 0
    no_ws = tensors.DecodeDevice(inp, plan, with_logits=False)
    _run_noalloc(plan, no_ws)
    torch.cuda.synchronize()
    for a, b in zip(_outputs(with_ws), _outputs(no_ws)):
        assert torch.equal(a, b)
    return plan, no_ws


def test_noalloc_matches_workspace_entry_point_twice():
    first = synth.decode_batch(rows=16)
    plan, dev = _compare(first)
    _check_oracle(first, dev, plan, oracle.reference_rows(first, rows=[0, 7, 15], mode="sparse"))
    second = synth.tiny_decode(0)  # other geometry, same scratch
    plan, dev = _compare(second)
    _check_oracle(second, dev, plan, oracle.reference_rows(second, mode="dense"))
    # back to the first shape: nothing left in the scratch changes the result
    plan = tensors.plan_for(first.geom, max_rows=first.rows)
    again = tensors.DecodeDevice(first, plan, with_logits=False)
    _run_noalloc(plan, again)
    ref = tensors.DecodeDevice(first, plan, with_logits=False)
    ref.run(plan)
    torch.cuda.synchronize()
    assert torch.equal(again.topk_out, ref.topk_out) and torch.equal(again.col_indices, ref.col_indices)


def test_noalloc_takes_exactly_what_its_scratch_holds():
    """The scratch holds the tile counters (4 bytes per plan row, rounded up to
    256) and rows x sparse columns x 4 bytes of logits. The largest row count
    that fits runs; one more row is refused and enqueues nothing."""
    inp = synth.decode_batch(rows=2)  # 4096 sparse columns
    plan = tensors.plan_for(inp.geom, max_rows=1024)
    counters = (4 * plan.max_rows + 255) // 256 * 256
    fit = (smq.SMQ_NOALLOC_SCRATCH_BYTES - counters) // (4 * plan.num_sparse_cols)
    assert fit == 511
    dev = plan.device
    H, D = inp.geom.num_heads, inp.geom.head_dim

    def buffers(rows):
        q = torch.zeros((rows, H, D), dtype=torch.uint8, device=dev)
        qs = torch.ones(rows, dtype=torch.float32, device=dev)
        w = torch.zeros((rows, H), dtype=torch.bfloat16, device=dev)
        ri = torch.zeros(rows, dtype=torch.int32, device=dev)
        ke = torch.ones(rows, dtype=torch.int32, device=dev)  # one position per row
        cand = torch.zeros((rows, plan.candidate_topk_blocks), dtype=torch.int32, device=dev)
        top = torch.full((rows, plan.topk), -7, dtype=torch.int32, device=dev)
        si = torch.full((rows, plan.num_sparse_blocks), -7, dtype=torch.int32, device=dev)
        end = torch.full((rows,), -7, dtype=torch.int32, device=dev)
        return q, qs, w, ri, ke, cand, top, si, end

    kc = torch.from_numpy(np.ascontiguousarray(inp.k_cache)).to(dev)
    bt = torch.from_numpy(np.ascontiguousarray(inp.block_table)).to(dev)
    q, qs, w, ri, ke, cand, top, si, end = buffers(fit)
    smq.sparse_mqa_logits_topk_decode_noalloc(plan, q, qs, w, kc, bt, ri, ke, cand, top, si, end)
    torch.cuda.synchronize()
    assert int((end == 1).sum()) == fit, "every row has its one position"
    assert bool((top[:, 0] == 0).all()) and bool((top[:, 1:] == -1).all()), "token 0, then -1"
    q, qs, w, ri, ke, cand, top, si, end = buffers(fit + 1)
    with pytest.raises(smq.SMQError) as e:
        smq.sparse_mqa_logits_topk_decode_noalloc(plan, q, qs, w, kc, bt, ri, ke, cand, top, si, end)
    assert e.value.code == smq.SMQ_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert int((top == -7).sum()) == top.numel() and int((end == -7).sum()) == fit + 1
