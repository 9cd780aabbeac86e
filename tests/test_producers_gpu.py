"""The device producers against the oracle, byte for byte: the MXFP4 K-cache
writer (sparse_mqa_write_k_cache) and the query quantiser
(sparse_mqa_quantize_q), called through the C ABI. The inputs include the
rounding's corner cases: elements on E2M1 / E4M3 midpoints, saturation,
groups of zeros, tiny values, negative values that round to zero."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300 import synth, tensors

from gpu_check import check_rows

pytestmark = pytest.mark.gpu

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _keys(rng, ntok):
    """bf16 keys whose 32-element groups take many scales, with midpoints, zeros and tiny values."""
    x = rng.standard_normal((ntok, 128)).astype(np.float32)
    x *= (2.0 ** rng.integers(-30, 30, size=(ntok, 4))).repeat(32, axis=1).astype(np.float32)
    mids = np.array([(E2M1[i] + E2M1[i + 1]) / 2 for i in range(7)], dtype=np.float32)
    for t in range(0, ntok, 5):  # groups whose elements sit on midpoints of their scale's grid
        g = int(rng.integers(0, 4))
        e = int(rng.integers(-10, 10))
        vals = rng.choice(np.concatenate([mids, -mids, [6.0, -6.0]]), size=32).astype(np.float32)
        vals[0] = 6.0  # amax exactly 6 * 2^e
        x[t, 32 * g:32 * g + 32] = vals * np.float32(2.0 ** e)
    x[3, :32] = 0.0                           # a group of zeros
    x[4, 32:64] = np.float32(1e-38)           # tiny values
    x[6, 64:96] = -np.float32(2.0 ** -5)      # negative values that round to -0 beside a large one
    x[6, 64] = 100.0
    x[7, 96:] = rng.standard_normal(32).astype(np.float32) * np.float32(1e30)  # a large scale
    return _bf16(x)


def test_k_cache_writer_matches_oracle():
    rng = np.random.Generator(np.random.PCG64(41))
    page, npages, ntok = 64, 24, 900
    plan = smq.Plan(num_heads=64, page_size=page, candidate_block_size=128, candidate_topk_blocks=8, topk=64,
                    max_rows=4)
    k = _keys(rng, ntok)
    slots = rng.permutation(page * npages)[:ntok].astype(np.int64)
    slots[rng.choice(ntok, 60, replace=False)] = -1
    cache0 = np.full((npages, plan.page_bytes), 0xA5, dtype=np.uint8)
    ref = cache0.copy()
    oracle.default().write_k_cache(k.view(torch.int16).numpy().view(np.uint16), slots, ref, page)
    dev = plan.device
    cache = torch.from_numpy(cache0).to(dev)
    ws = plan.workspace(1)
    smq.sparse_mqa_write_k_cache(plan, k.to(dev), torch.from_numpy(slots).to(dev), cache, ws)
    assert smq.smq_get_status(ws) == 0
    got = cache.cpu().numpy()
    bad = np.argwhere(got != ref)
    assert len(bad) == 0, f"{len(bad)} cache bytes differ; first at page/byte {bad[:4].tolist()}"


def test_k_cache_writer_reports_a_slot_past_the_cache():
    plan = smq.Plan(num_heads=64, page_size=64, candidate_block_size=128, candidate_topk_blocks=8, topk=64,
                    max_rows=4)
    dev = plan.device
    rng = np.random.Generator(np.random.PCG64(43))
    k = _bf16(rng.standard_normal((3, 128)))
    slots = torch.tensor([5, 4 * 64 + 1, 70], dtype=torch.int64, device=dev)  # the middle one is past 4 pages
    cache = torch.zeros((4, plan.page_bytes), dtype=torch.uint8, device=dev)
    ws = plan.workspace(1)
    smq.sparse_mqa_write_k_cache(plan, k.to(dev), slots, cache, ws)
    assert smq.smq_get_status(ws) & smq.SMQ_ERR_BOUNDS
    ref = np.zeros((4, plan.page_bytes), dtype=np.uint8)
    kk = k.view(torch.int16).numpy().view(np.uint16)
    oracle.default().write_k_cache(kk[[0, 2]], np.array([5, 70], dtype=np.int64), ref, 64)
    assert np.array_equal(cache.cpu().numpy(), ref), "the other tokens are written"


@pytest.mark.parametrize("heads", [8, 64, 128])
def test_q_quantiser_matches_oracle(heads):
    rng = np.random.Generator(np.random.PCG64(47 + heads))
    rows = 37
    x = rng.standard_normal((rows, heads, 128)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-4, 4, size=rows)).astype(np.float32)[:, None, None]
    x[5] = 0.0  # a zero row: scale 1
    # a row whose amax is 448 (scale 1) with elements on E4M3 midpoints
    e4 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    mids = ((e4[:-1] + e4[1:]) / 2).astype(np.float32)
    row = rng.choice(np.concatenate([mids, -mids]), size=heads * 128).astype(np.float32)
    row[0] = 448.0
    x[9] = row.reshape(heads, 128)
    w = (rng.standard_normal((rows, heads)) * 0.3).astype(np.float32)
    w[0, :4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e-39]  # bf16 ties, a subnormal
    qb = _bf16(x)
    q8_ref, sc_ref, wb_ref = oracle.default().quantize_q(qb.view(torch.int16).numpy().view(np.uint16), w)
    plan = smq.Plan(num_heads=heads, page_size=64, candidate_block_size=128, candidate_topk_blocks=8, topk=64,
                    max_rows=rows)
    dev = plan.device
    q8 = torch.empty((rows, heads, 128), dtype=torch.uint8, device=dev)
    sc = torch.empty(rows, dtype=torch.float32, device=dev)
    wb = torch.empty((rows, heads), dtype=torch.int16, device=dev)
    smq.sparse_mqa_quantize_q(plan, qb.to(dev), torch.from_numpy(w).to(dev), q8, sc, wb)
    torch.cuda.synchronize()
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32)), "scales"
    got = q8.cpu().numpy()
    bad = np.argwhere(got != q8_ref)
    assert len(bad) == 0, f"{len(bad)} E4M3 codes differ; first {bad[:4].tolist()}"
    assert np.array_equal(wb.cpu().numpy().view(np.uint16), wb_ref), "bf16 weights"


def test_produced_inputs_through_the_decode_call():
    """Keys and queries quantised on the device feed the decode call; its
    results match the oracle on those bytes."""
    rng = np.random.Generator(np.random.PCG64(53))
    base = synth.decode_batch(rows=8)  # shapes, tables and candidates
    g = base.geom
    plan = tensors.plan_for(g, max_rows=base.rows)
    dev = plan.device
    npages = base.k_cache.shape[0]
    ntok = npages * g.page_size
    k = _bf16(rng.standard_normal((ntok, 128)))
    cache = torch.zeros((npages, plan.page_bytes), dtype=torch.uint8, device=dev)
    ws = plan.workspace(base.rows)
    smq.sparse_mqa_write_k_cache(plan, k.to(dev), torch.arange(ntok, dtype=torch.int64, device=dev), cache, ws)
    qb = _bf16(rng.standard_normal((base.rows, g.num_heads, 128)))
    w = (rng.standard_normal((base.rows, g.num_heads)) / 8).astype(np.float32)
    q8 = torch.empty((base.rows, g.num_heads, 128), dtype=torch.uint8, device=dev)
    sc = torch.empty(base.rows, dtype=torch.float32, device=dev)
    wb = torch.empty((base.rows, g.num_heads), dtype=torch.int16, device=dev)
    smq.sparse_mqa_quantize_q(plan, qb.to(dev), torch.from_numpy(w).to(dev), q8, sc, wb)
    torch.cuda.synchronize()
    inp = synth.DecodeInputs(g, q8.cpu().numpy(), sc.cpu().numpy(), wb.cpu().numpy().view(np.uint16),
                             cache.cpu().numpy(), base.block_table, base.row_indices, base.row_ke,
                             base.candidate_blocks)
    d = tensors.DecodeDevice(inp, plan)
    d.run(plan)
    assert smq.smq_get_status(d.workspace) == 0
    check_rows(inp, d, plan, oracle.reference_rows(inp, mode="sparse"))
