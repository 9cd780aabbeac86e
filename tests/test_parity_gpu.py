"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every row against the dense oracle (score the whole
context, mask, sort).  Full-size workloads compare every row's expansion,
logits and top-k set against the oracle's candidate-only mode (equal to the
dense mode by the pinned invariant), in the launch configuration the
benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import synth, tensors

from gpu_check import check_rows, run_decode, run_prefill

pytestmark = pytest.mark.gpu


def _ok(status):
    assert status == 0, f"device status {status}"


def test_tiny_decode_dense():
    inp = synth.tiny_decode(0)
    plan, dev, status = run_decode(inp, with_logits_bf16=True)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense"))


GEOMS = [
    # heads, page, cbs, ncb, topk, ctx range
    (8, 64, 64, 6, 100, (1, 700)),
    (16, 16, 32, 9, 40, (30, 900)),
    (32, 32, 128, 5, 500, (100, 2000)),
    (64, 128, 256, 4, 300, (1, 3000)),
    (64, 64, 128, 16, 2048, (2048, 6000)),
    (72, 64, 64, 8, 128, (64, 1100)),
    (128, 64, 128, 7, 512, (1, 2500)),
    (128, 32, 64, 12, 64, (500, 1500)),
    # more than 64 candidate blocks: expansion and top-k in their own kernels (16384 columns)
    (64, 64, 128, 128, 2048, (14000, 20000)),
    # 8448 columns: too wide for a row cluster; the persistent kernel expands and selects itself
    (64, 64, 256, 33, 300, (5000, 9000)),
]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"H{g[0]}-p{g[1]}-cbs{g[2]}-ncb{g[3]}-k{g[4]}")
def test_decode_geometries_dense(geom):
    h, page, cbs, ncb, topk, (lo, hi) = geom
    rng = np.random.Generator(np.random.PCG64(h * 1000 + page + cbs))
    rows = 12
    ctx = rng.integers(lo, hi + 1, size=rows)
    inp = synth._paged_decode(seed=h + page, rows=rows, h=h, page_size=page, cbs=cbs, ncb=ncb, topk=topk,
                              ctx=ctx, row_perm=True)
    plan, dev, status = run_decode(inp, with_logits_bf16=True)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense"))


ADVERSARIAL_KINDS = ["mixed", "lone", "none", "mixed", "lone", "mixed", "mixed"]


@pytest.mark.parametrize("ncb,rows", [(24, 14), (32, 14), (33, 14), (56, 14), (64, 14), (40, 90), (80, 14)],
                         ids=lambda v: str(v))
def test_expansion_of_repeated_negative_and_out_of_range_ids(ncb, rows):
    """Decode rows with at most 64 candidate blocks are expanded inside the
    score kernel: the first 32 ids by a warp match, the next 32 against the
    first. Candidate rows with ids repeated inside a half and across the
    halves, -1 and other negative ids (down to INT32_MIN), blocks at and far
    past the row end (up to INT32_MAX), a row whose one in-range block
    repeats, rows with no in-range block and a row of zero context must give
    the oracle's expansion exactly, its logits and its top-k sets. 90 rows
    take the separate top-k kernel; 80 blocks take the expansion kernel."""
    cbs, page, topk = 64, 64, 256
    rng = np.random.Generator(np.random.PCG64(1000 + ncb + rows))
    ctx = rng.integers(1, 3000, size=rows)
    ctx[1] = 0
    ctx[2] = 65  # two blocks, the second holds one position

    def cand_fn(g, r, L):
        return synth.adversarial_blocks(g, ncb, L, cbs, ADVERSARIAL_KINDS[r % len(ADVERSARIAL_KINDS)])

    inp = synth._paged_decode(seed=77 + ncb, rows=rows, h=64, page_size=page, cbs=cbs, ncb=ncb, topk=topk,
                              ctx=ctx, cand_fn=cand_fn, row_perm=True)
    cand = inp.candidate_blocks
    assert (cand < -1).any() and (cand == -1).any()
    assert any(len(set(c[c >= 0].tolist())) < int((c >= 0).sum()) for c in cand)
    plan, dev, status = run_decode(inp)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense"))


def test_prefill_expansion_of_repeated_negative_and_out_of_range_ids():
    """The prefill call's expansion kernel on the same adversarial candidate rows."""
    cbs, ncb = 64, 20

    def cand_fn(g, r, L):
        return synth.adversarial_blocks(g, ncb, L, cbs, ADVERSARIAL_KINDS[r % len(ADVERSARIAL_KINDS)])

    inp = synth.prefill_chunk(seed=31, seq_lens=(900, 1300), queries_per_seq=21, num_heads=32, page_size=64,
                              cbs=cbs, ncb=ncb, topk=150, cand_fn=cand_fn)
    plan, dev, status = run_prefill(inp)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense", contig=(kv, ks)))


@pytest.mark.parametrize("next_n,requests", [(2, 12), (4, 9), (3, 60)])
def test_multi_token_decode_rows(next_n, requests):
    """next_n query tokens per request (speculative decoding): the rows of a
    request share its block-table row through row_indices, and each sees its
    own causal context. 180 rows take the persistent kernel and the top-k
    kernel; fewer take one cluster per row."""
    inp = synth.multi_token_decode(seed=60 + next_n, requests=requests, next_n=next_n, ctx_range=(300, 6000),
                                   ncb=12, topk=500)
    assert len(set(inp.row_indices.tolist())) == requests and inp.block_table.shape[0] == requests
    plan, dev, status = run_decode(inp, with_logits_bf16=True)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense"))


def test_decode_batch_full_size():
    """64 rows, H=64, contexts 4096..32768, 32 blocks of 128, topk 2048."""
    inp = synth.decode_batch()
    plan, dev, status = run_decode(inp)
    _ok(status)
    ref = oracle.reference_rows(inp, mode="sparse")
    check_rows(inp, dev, plan, ref)
    dense = oracle.reference_rows(inp, rows=[0, 1], mode="dense")
    check_rows(inp, dev, plan, dense, all_rows=False)


def test_long_context_full_size():
    """256 rows, contexts log-uniform to 131072, 10% shorter than topk: every
    row against the oracle's candidate-only mode."""
    inp = synth.long_context_decode()
    plan, dev, status = run_decode(inp)
    _ok(status)
    assert any(inp.row_ke[r] < inp.geom.topk for r in range(inp.rows))
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="sparse"))


def test_prefill_small_dense():
    inp = synth.prefill_chunk(seed=12, seq_lens=(1500, 2300, 700), queries_per_seq=40, num_heads=64,
                              page_size=64, cbs=128, ncb=6, topk=300)
    plan, dev, status = run_prefill(inp, with_logits_bf16=True)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    assert np.array_equal(tensors.to_numpy(dev.k_values), kv)
    assert np.array_equal(tensors.to_numpy(dev.k_scales), ks)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense", contig=(kv, ks)))


def test_prefill_unaligned_sequence_starts():
    """Sequence starts that are not multiples of 4 positions exercise the
    scale loads that begin below the row and index past the remainder."""
    inp = synth.prefill_chunk(seed=5, seq_lens=(1021, 999, 1502), queries_per_seq=24, num_heads=16,
                              page_size=32, cbs=64, ncb=9, topk=200)
    assert any(int(s) % 4 for s in inp.cu_seq_lens[1:-1])
    plan, dev, status = run_prefill(inp)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense", contig=(kv, ks)))


@pytest.mark.parametrize("seq_lens,page,cbs,ncb,seed", [
    ((1021, 999, 1502), 32, 64, 9, 31),    # 4 slots per window, two per block; unaligned starts
    ((2000, 1777), 64, 256, 5, 32),        # a block spans two windows
    ((900, 1300, 517), 16, 16, 40, 33),    # 8 slots per window, one per block
])
def test_window_major_prefill_matches_the_row_major_path(seq_lens, page, cbs, ncb, seed):
    """The window-major prefill (rows grouped by the 128-key windows they
    selected, two rows per MMA) gives the row-major kernel's logits and ids
    bit for bit, and both match the oracle; windows hold partial slot masks,
    sequence starts are not multiples of 128 and windows run past the end of
    the workspace."""
    inp = synth.prefill_chunk(seed=seed, seq_lens=seq_lens, queries_per_seq=30, num_heads=64, page_size=page,
                              cbs=cbs, ncb=ncb, topk=150)
    plan, wm, status = run_prefill(inp, window_major=True)
    _ok(status)
    _, rm, status = run_prefill(inp, plan=plan, window_major=False)
    _ok(status)
    assert torch.equal(wm.sparse_indices, rm.sparse_indices) and torch.equal(wm.end, rm.end)
    valid = torch.arange(plan.num_sparse_cols, device=wm.end.device)[None, :] < wm.end[:, None].long()
    assert torch.equal(wm.logits[valid], rm.logits[valid])
    assert torch.equal(wm.topk_out, rm.topk_out)
    kv, ks = oracle.gather_reference(inp)
    check_rows(inp, wm, plan, oracle.reference_rows(inp, mode="dense", contig=(kv, ks)))


def test_prefill_rows_through_the_paged_decode_call():
    """In-place paged prefill: the chunk's rows, run through the paged decode
    call on the cache itself, give the gather path's expansion, logits and ids."""
    inp = synth.prefill_chunk(seed=12, seq_lens=(1500, 2300, 700), queries_per_seq=40, num_heads=64,
                              page_size=64, cbs=128, ncb=6, topk=300)
    plan, dev, status = run_prefill(inp)
    _ok(status)
    dec = synth.prefill_as_decode(inp)
    plan_d, ddev, status_d = run_decode(dec)
    _ok(status_d)
    assert torch.equal(ddev.sparse_indices, dev.sparse_indices) and torch.equal(ddev.end, dev.end)
    valid = torch.arange(plan.num_sparse_cols, device=dev.end.device)[None, :] < dev.end[:, None].long()
    assert torch.equal(ddev.logits[valid], dev.logits[valid])
    assert torch.equal(ddev.topk_out, dev.topk_out)
    check_rows(dec, ddev, plan_d, oracle.reference_rows(dec, rows=range(0, dec.rows, 7), mode="sparse"),
               all_rows=False)


def test_prefill_chunk_full_size():
    """4096 rows from 2 sequences (28672 + 36864), causal ranges, topk 2048:
    every row against the oracle's candidate-only mode."""
    inp = synth.prefill_chunk()
    plan, dev, status = run_prefill(inp)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    assert np.array_equal(tensors.to_numpy(dev.k_values), kv)
    assert np.array_equal(tensors.to_numpy(dev.k_scales), ks)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="sparse", contig=(kv, ks)))


def test_shared_schedule_reuse_is_bit_identical():
    """4 consumer layers share one expansion: reusing it gives the same bytes
    as expanding inside every call."""
    layers = synth.shared_schedule_layers(layers=4)
    plan = tensors.plan_for(layers[0].geom, max_rows=layers[0].rows)
    devs = [tensors.DecodeDevice(inp, plan) for inp in layers]
    devs[0].expand(plan)
    for d in devs[1:]:
        d.sparse_indices.copy_(devs[0].sparse_indices)
        d.end.copy_(devs[0].end)
    for d in devs:
        d.run(plan, expansion_ready=True)
    fresh = [tensors.DecodeDevice(inp, plan) for inp in layers]
    for d in fresh:
        d.run(plan, expansion_ready=False)
    for d in devs + fresh:
        _ok(smq.smq_get_status(d.workspace))
    for a, b in zip(devs, fresh):
        assert torch.equal(a.topk_out, b.topk_out)
        assert torch.equal(a.logits, b.logits)
        assert torch.equal(a.sparse_indices, b.sparse_indices) and torch.equal(a.end, b.end)
    for li, inp in enumerate(layers):
        check_rows(inp, devs[li], plan, oracle.reference_rows(inp, mode="sparse"))


def test_expand_golden_cases_on_gpu():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "expansion_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        page = c["sbkv"]
        ncb = len(c["cand"])
        plan = smq.Plan(num_heads=8, page_size=page, candidate_block_size=c["cbs"], candidate_topk_blocks=ncb,
                        topk=1, max_rows=1, sparse_block_kv=c["sbkv"])
        assert plan.num_sparse_blocks == c["nsb"] == ncb * c["cbs"] // c["sbkv"]
        cand = torch.tensor([c["cand"]], dtype=torch.int32, device="cuda")
        ke = torch.tensor([c["L"]], dtype=torch.int32, device="cuda")
        si = torch.full((1, c["nsb"]), -7, dtype=torch.int32, device="cuda")
        end = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        ws = plan.workspace(1)
        smq.sparse_mqa_candidate_expand(plan, cand, None, ke, si, end, ws)
        assert si.cpu().tolist()[0] == c["sparse_indices"], c["name"]
        assert int(end.item()) == c["end"], c["name"]


def test_ties_any_k_subset():
    """Every key equal: all valid logits tie, any k of them is correct."""
    inp = synth.tiny_decode(0)
    inp.k_cache[:, : 64 * 64] = 0x22  # every element 1.0
    inp.k_cache[:, 64 * 64:] = 127
    plan, dev, status = run_decode(inp)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="dense"))


def test_two_values_many_ties():
    """Keys of two values only: the logits take a few distinct values, each
    shared by many columns, so the top-k threshold falls inside a crowded bin
    (ties ranked by column, or the radix passes when the bin overflows)."""
    inp = synth.decode_batch(rows=8)
    half = inp.geom.page_size * 64
    inp.k_cache[:, :half] = 0x22  # every element 1.0
    inp.k_cache[::3, :half] = 0x44  # every third page 3.0
    inp.k_cache[:, half:] = 127
    plan, dev, status = run_decode(inp)
    _ok(status)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, rows=range(8), mode="sparse"))


@pytest.mark.parametrize("mode", ["equal", "two_values"])
def test_prefill_topk_kernel_with_ties(mode):
    """The separate top-k kernel (prefill rows) on crowded thresholds: every
    key equal (the value range is a single point) or keys of two values (the
    threshold bin overflows and the digit passes decide); ties go by column."""
    inp = synth.prefill_chunk(seed=41, seq_lens=(1500, 2300), queries_per_seq=30, num_heads=64, page_size=64,
                              cbs=128, ncb=8, topk=300)
    half = inp.geom.page_size * 64
    inp.k_cache[:, :half] = 0x22  # every element 1.0
    if mode == "two_values":
        inp.k_cache[::3, :half] = 0x44  # every third page 3.0
    inp.k_cache[:, half:] = 127
    plan, dev, status = run_prefill(inp)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="sparse", contig=(kv, ks)))


def test_prefill_topk_sampled_range_cases():
    """The warp top-k bins each row over the value range of its first 128
    columns. Every other page of the cache holds equal keys, so across the
    rows: a first candidate block of equal keys (the sample has no spread and
    the exact range is taken), many equal keys outside the sampled range (the
    threshold bin overflows and the digit passes decide), ties by column."""
    inp = synth.prefill_chunk(seed=43, seq_lens=(1500, 2300), queries_per_seq=30, num_heads=64, page_size=64,
                              cbs=128, ncb=8, topk=300)
    half = inp.geom.page_size * 64
    inp.k_cache[0::2, :half] = 0x22  # every element 1.0 on even pages
    inp.k_cache[0::2, half:] = 127
    plan, dev, status = run_prefill(inp)
    _ok(status)
    kv, ks = oracle.gather_reference(inp)
    check_rows(inp, dev, plan, oracle.reference_rows(inp, mode="sparse", contig=(kv, ks)))


def test_zero_rows_is_a_no_op():
    inp = synth.tiny_decode(0)
    plan = tensors.plan_for(inp.geom, max_rows=4)
    dev = tensors.DecodeDevice(inp, plan)
    empty = torch.empty((0,) + tuple(dev.q.shape[1:]), dtype=torch.uint8, device=plan.device)
    smq.sparse_mqa_logits_topk_decode(plan, empty, dev.q_scale[:0], dev.weights[:0], dev.k_cache, dev.block_table,
                                      dev.row_indices[:0], dev.row_ke[:0], dev.candidate_blocks[:0],
                                      dev.topk_out[:0], dev.sparse_indices[:0], dev.end[:0], dev.workspace)
    torch.cuda.synchronize()
    assert int((dev.topk_out == -7).sum()) == dev.topk_out.numel()


def test_out_of_range_page_sets_bounds_status():
    """A corrupt block-table entry is reported, not read."""
    inp = synth.tiny_decode(0)
    req = int(inp.row_indices[0])
    b = int(inp.candidate_blocks[0][0])
    inp.block_table[req][b] = inp.k_cache.shape[0] + 5
    plan, dev, status = run_decode(inp)
    assert status & smq.SMQ_ERR_BOUNDS
    # rows that never touch the corrupt entry are unaffected
    ref = oracle.reference_rows(inp, rows=[1, 2, 3], mode="dense")
    check_rows(inp, dev, plan, ref, all_rows=False)


def test_repeat_calls_are_deterministic():
    inp = synth.decode_batch(rows=16)
    plan, dev, status = run_decode(inp)
    _ok(status)
    first = (dev.topk_out.clone(), dev.logits.clone())
    dev.run(plan)
    _ok(smq.smq_get_status(dev.workspace))
    assert torch.equal(first[0], dev.topk_out) and torch.equal(first[1], dev.logits)


def test_prepared_call_matches_the_plain_call():
    """DecodeCall marshals the arguments once; each call must give the plain
    call's bytes, also after the inputs are rewritten in place."""
    inp = synth.decode_batch(rows=16)
    plan, dev, status = run_decode(inp)
    _ok(status)
    ref = (dev.topk_out.clone(), dev.logits.clone())
    call = smq.DecodeCall(plan, dev.q, dev.q_scale, dev.weights, dev.k_cache, dev.block_table, dev.row_indices,
                          dev.row_ke, dev.candidate_blocks, dev.topk_out, dev.sparse_indices, dev.end, dev.workspace,
                          col_indices=dev.col_indices, logits_out=dev.logits)
    dev.topk_out.fill_(-7)
    call()
    _ok(smq.smq_get_status(dev.workspace))
    assert torch.equal(dev.topk_out, ref[0]) and torch.equal(dev.logits, ref[1])
    # new queries and weights written into the same buffers
    import copy
    fresh = synth.decode_batch(seed=9, rows=16)
    other = copy.copy(inp)
    other.q, other.q_scale, other.weights = fresh.q, fresh.q_scale, fresh.weights
    other_dev = tensors.DecodeDevice(other, plan)
    for name in ("q", "q_scale", "weights"):
        getattr(dev, name).copy_(getattr(other_dev, name))
    call()
    _ok(smq.smq_get_status(dev.workspace))
    other_dev.run(plan)
    _ok(smq.smq_get_status(other_dev.workspace))
    assert not torch.equal(dev.topk_out, ref[0])
    assert torch.equal(dev.topk_out, other_dev.topk_out) and torch.equal(dev.logits, other_dev.logits)


def test_tile_counters_are_left_at_zero():
    """Rows whose top-k the score kernel selects count finished tiles in the
    workspace; a call leaves those counters at zero for the next call."""
    inp = synth.decode_batch(rows=16)
    plan, dev, status = run_decode(inp)
    _ok(status)
    counters = dev.workspace[256:256 + 4 * plan.max_rows].view(torch.int32)
    assert int(counters.abs().sum()) == 0
    dev.run(plan)
    _ok(smq.smq_get_status(dev.workspace))
    assert int(counters.abs().sum()) == 0
    check_rows(inp, dev, plan, oracle.reference_rows(inp, rows=[0, 5, 15], mode="sparse"))
