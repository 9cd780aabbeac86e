"""Run the CUDA path through the C ABI and compare it with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import check
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import tensors


def _token_of(si_row, c, sbkv):
    return si_row[c // sbkv] * sbkv + c % sbkv


def check_rows(inp, dev, plan, ref_rows, all_rows=True):
    """Compare GPU outputs with oracle RowResults (dict row -> RowResult).

    Rows in ref_rows get the full comparison (expansion, every logit, the
    top-k set).  With all_rows, every other row still gets the exact
    expansion check and the structural top-k checks (count, distinct,
    candidate columns only, col_indices consistent)."""
    g = inp.geom
    k = g.topk
    sbkv = plan.sparse_block_kv
    si = tensors.to_numpy(dev.sparse_indices)
    end = tensors.to_numpy(dev.end)
    top = tensors.to_numpy(dev.topk_out)
    cols = tensors.to_numpy(dev.col_indices)
    logits = tensors.to_numpy(dev.logits)
    nsb = plan.num_sparse_blocks
    rows = range(inp.rows) if all_rows else sorted(ref_rows)
    orc = oracle.default()
    l16 = getattr(dev, "logits_bf16", None)
    if l16 is not None:
        # each bf16 logit is the call's own fp32 logit rounded to nearest even (torch's cast), -inf past end
        assert logits is not None, "the bf16 logits are compared with the fp32 ones of the same call"
        f32 = dev.logits
        valid = torch.arange(f32.shape[1], device=f32.device)[None, :] < dev.end[:, None].long()
        expect = f32.to(torch.bfloat16).view(torch.int16)
        assert torch.equal(l16[valid], expect[valid]), "bf16 logits are the fp32 logits rounded to nearest even"
        assert bool((l16[~valid] == -128).all()), "masked bf16 logits are -inf (0xFF80)"
        l16 = l16.view(torch.bfloat16).to(torch.float64).cpu().numpy()
    for r in rows:
        if hasattr(inp, "row_ke"):
            L = int(inp.row_ke[r])
        else:
            L = int(inp.cu_seqlen_ke[r]) - int(inp.cu_seqlen_ks[r])
        esi, eend = orc.expand(g.candidate_block_size, sbkv, inp.candidate_blocks[r], max(L, 0), nsb)
        assert np.array_equal(si[r], esi), f"row {r}: sparse_indices {si[r][:8]} vs {esi[:8]}"
        assert end[r] == eend, f"row {r}: end {end[r]} vs {eend}"
        e = int(end[r])
        want = min(k, e)
        assert np.all(top[r, want:] == -1), f"row {r}: -1 padding"
        sel = top[r, :want]
        assert np.all(sel >= 0) and len(np.unique(sel)) == want, f"row {r}: ids"
        positions = oracle._columns(esi, e, sbkv)
        assert np.all(np.isin(sel, positions)), f"row {r}: ids outside candidates"
        if cols is not None:
            assert np.all(cols[r, want:] == -1)
            assert np.array_equal(np.array([_token_of(si[r], c, sbkv) for c in cols[r, :want]]), sel), \
                f"row {r}: col_indices do not map to the ids"
        if logits is not None:
            assert np.all(np.isneginf(logits[r, e:])), f"row {r}: masked columns must be -inf"
        if r in ref_rows:
            row = ref_rows[r]
            ref_logits = row.logits[row.positions] if row.valid is not None else row.logits
            check.check_logits(logits[r, :e], ref_logits, f"row {r} logits")
            if l16 is not None:
                check.check_logits_bf16(l16[r, :e], ref_logits, f"row {r} bf16 logits")
            check.check_topk(top[r], row, k, f"row {r} top-k")


def run_decode(inp, plan=None, **kw):
    plan = plan or tensors.plan_for(inp.geom, max_rows=max(inp.rows, 1))
    dev = tensors.DecodeDevice(inp, plan, **kw)
    dev.run(plan)
    status = smq.smq_get_status(dev.workspace)
    return plan, dev, status


def run_prefill(inp, plan=None, **kw):
    plan = plan or tensors.plan_for(inp.geom, max_rows=max(inp.rows, 1))
    dev = tensors.PrefillDevice(inp, plan, **kw)
    dev.gather(plan)
    dev.run(plan)
    status = smq.smq_get_status(dev.workspace)
    return plan, dev, status
