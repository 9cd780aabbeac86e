"""The candidate-source indexer (sparse_mqa_candidate_source_decode) against
the oracle: dense logits over each row's context, every block's maximum and
the row's published blocks. The published list is a decision that floating
point takes, so it is checked twice: exactly, against the oracle's selection
applied to the GPU's own block scores; and as a set against the oracle's
float64 selection, where only blocks tied within the logit tolerance at the
last published score may differ."""

import numpy as np
import pytest
import torch

import oracle
from oracle import check
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import synth, tensors

from gpu_check import check_rows, run_decode

pytestmark = pytest.mark.gpu


def _run_source(inp, plan, max_context):
    dev = plan.device
    d = tensors.DecodeDevice(inp, plan, with_logits=False, with_cols=False)
    nblk = -(-max_context // inp.geom.candidate_block_size)
    cand = torch.full((inp.rows, inp.geom.candidate_topk_blocks), -7, dtype=torch.int32, device=dev)
    scores = torch.full((inp.rows, nblk), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(smq.smq_source_workspace_size(plan, inp.rows, max_context), dtype=torch.uint8, device=dev)
    smq.smq_workspace_init(plan, ws)
    smq.sparse_mqa_candidate_source_decode(plan, d.q, d.q_scale, d.weights, d.k_cache, d.block_table,
                                           d.row_indices, d.row_ke, max_context, cand, ws, block_scores=scores)
    status = smq.smq_get_status(ws)
    return cand.cpu().numpy(), scores.cpu().numpy(), status


def _check_source(inp, cand, scores):
    g = inp.geom
    orc = oracle.default()
    ref = oracle.source_rows(inp)
    for r in range(inp.rows):
        rc, rs, _ = ref[r]
        nb = len(rs)
        check.check_logits(scores[r, :nb], rs, f"row {r} block scores")
        assert np.all(np.isneginf(scores[r, nb:])), f"row {r}: scores past the row's blocks are -inf"
        # exact: the oracle's rule on the GPU's own scores
        mine, _ = orc.source_blocks(scores[r, :nb].astype(np.float64), 1, g.candidate_topk_blocks)
        assert np.array_equal(cand[r], mine), f"row {r}: {cand[r][:8]} vs {mine[:8]}"
        # as a set against the float64 selection: differences only between near-ties
        n = min(nb, g.candidate_topk_blocks)
        assert np.all(cand[r, n:] == -1)
        diff = np.setxor1d(cand[r, :n], rc[:n])
        if len(diff):
            v_k = rs[rc[n - 1]]
            for b in diff.tolist():
                assert abs(rs[b] - v_k) <= max(check.ATOL, check.RTOL * abs(v_k)), \
                    f"row {r}: block {b} (score {rs[b]}) is not tied with the last published ({v_k})"


def test_source_on_decode_rows():
    inp = synth.decode_batch(seed=71, rows=12)
    inp.row_ke[3] = 1000   # 8 blocks: fewer than the 32 published, -1 after them
    inp.row_ke[5] = 0      # no context at all
    inp.row_ke[7] = 4097   # a last block of one position
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    max_context = int(inp.row_ke.max())
    cand, scores, status = _run_source(inp, plan, max_context)
    assert status == 0
    assert np.all(cand[5] == -1) and np.all(cand[3, 8:] == -1)
    _check_source(inp, cand, scores)


def test_source_on_long_contexts():
    inp = synth.long_context_decode(seed=73, rows=10)
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    cand, scores, status = _run_source(inp, plan, int(inp.row_ke.max()))
    assert status == 0
    _check_source(inp, cand, scores)


def test_source_then_consumer():
    """Two-level selection end to end: the source's blocks are the consumer
    call's candidates; the consumer's results match the oracle's on them."""
    inp = synth.decode_batch(seed=79, rows=16)
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    cand, scores, status = _run_source(inp, plan, int(inp.row_ke.max()))
    assert status == 0
    inp.candidate_blocks = cand.astype(np.int32)
    plan2, dev, status = run_decode(inp, plan=plan)
    assert status == 0
    check_rows(inp, dev, plan2, oracle.reference_rows(inp, mode="sparse"))


def test_source_context_past_the_bound_is_reported():
    inp = synth.decode_batch(seed=83, rows=4)
    plan = tensors.plan_for(inp.geom, max_rows=inp.rows)
    _, _, status = _run_source(inp, plan, int(inp.row_ke.max()) - 300)
    assert status & smq.SMQ_ERR_BOUNDS
