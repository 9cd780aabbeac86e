"""Pins of the CPU oracle: checks against facts that do not come from the
oracle itself.  Each pin takes an ``oracle.Oracle`` handle and raises
AssertionError on a mismatch, so the same pins also run against copies of
the oracle with a planted mistake (tests/test_oracle_mutants.py).

What pins what:
  e4m3 / bf16 decoders     every code vs torch's float8_e4m3fn / bfloat16 casts
  e2m1 / ue8m0 decoders    the OCP MX v1.0 value table; 2^(e-127) by ldexp
  one_hot                  closed form L[p] = max(0, K[p, d*]) through a
                           permuted block table: nibble order, group index,
                           page walk, token offset, ReLU
  relu_sign                closed form with two heads of opposite weight
  exact_rational           exact Fraction arithmetic on a tiny random case
  numpy_einsum             float64 einsum over tensors decoded with
                           independent tables (paged and contiguous K)
  monotone_topk            K increasing with position -> the k largest
                           valid positions; masking of -1, out-of-range and
                           repeated blocks
  ties                     all-equal keys -> the k smallest valid positions
  padding                  fewer valid positions than k -> those, then -1
  expansion_golden         hand-derived cases in golden/expansion_cases.json
  gather                   numpy slicing of the page bytes
  dense_equals_sparse      the invariant "candidate-only == dense-then-mask"
"""

from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle as oracle_pkg
from sparse_attention_top_expand_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# OCP MX v1.0, FP4 E2M1 value table, codes 0..7 (8..15 are the negatives).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
BF16_ONE = 0x3F80
E4M3_ONE = 0x38
E4M3_TWO = 0x40


def _e2m1(code):
    v = E2M1_TABLE[code & 7]
    return -v if code & 8 else v


# -------------------------------------------------------------- decoders


def pin_e4m3(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), f"e4m3 code {c:#x} should be NaN"
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), \
                f"e4m3 code {c:#x}: {got} != {ref[c]}"


def pin_bf16(orc):
    bits = np.arange(0, 65536, 97, dtype=np.int64).tolist() + [0x0000, 0x8000, 0x3F80, 0x7F7F, 0x0001, 0x807F]
    t = torch.tensor(bits, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    for b, ref in zip(bits, t):
        got = orc.bf16(b)
        if math.isnan(ref):
            assert math.isnan(got)
        else:
            assert got == ref, f"bf16 {b:#06x}: {got} != {ref}"


def pin_e2m1(orc):
    for c in range(16):
        assert orc.e2m1(c) == _e2m1(c), f"e2m1 {c}: {orc.e2m1(c)} != {_e2m1(c)}"
        assert math.copysign(1, orc.e2m1(c)) == (-1 if c & 8 else 1)


def pin_ue8m0(orc):
    for e in range(255):
        assert orc.ue8m0(e) == math.ldexp(1.0, e - 127), f"ue8m0 {e}"
    assert math.isnan(orc.ue8m0(255))


# -------------------------------------------------------------- closed forms


def _blank_decode(h, page, npages, L, ncb, cbs, topk, seed=5):
    """A decode input with every value zero, one request, a permuted table."""
    rng = np.random.Generator(np.random.PCG64(seed))
    d = synth.HEAD_DIM
    geom = synth.Geometry(h, d, page, cbs, ncb, topk)
    pb = synth.page_bytes(page, d)
    cache = np.zeros((npages, pb), dtype=np.uint8)
    cache[:, page * d // 2:] = 127  # unit scales
    bt = rng.permutation(npages).astype(np.int32)[None, :]
    q = np.zeros((1, h, d), dtype=np.uint8)
    qs = np.ones(1, dtype=np.float32)
    w = np.full((1, h), BF16_ONE, dtype=np.uint16)
    cand = np.full((1, ncb), -1, dtype=np.int32)
    return synth.DecodeInputs(geom, q, qs, w, cache, bt, np.zeros(1, np.int32),
                              np.array([L], np.int32), cand)


def _set_key(inp, p, d, nibble, scale_code):
    """Write element d of position p's key (through the request's table)."""
    g = inp.geom
    page = int(inp.block_table[0][p // g.page_size])
    tok = p % g.page_size
    byte_off = tok * (g.head_dim // 2) + d // 2
    b = int(inp.k_cache[page, byte_off])
    if d % 2 == 0:
        b = (b & 0xF0) | nibble
    else:
        b = (b & 0x0F) | (nibble << 4)
    inp.k_cache[page, byte_off] = b
    inp.k_cache[page, g.page_size * g.head_dim // 2 + tok * (g.head_dim // 32) + d // 32] = scale_code


def pin_one_hot(orc):
    """H=1, w=1, Q one-hot at d* equal to 1 => L[p] = max(0, K[p, d*])."""
    page, npages, L = 16, 8, 120
    for dstar, (qcode, qscale) in [(0, (E4M3_ONE, 1.0)), (1, (E4M3_TWO, 0.5)), (31, (E4M3_ONE, 1.0)),
                                   (32, (E4M3_TWO, 0.5)), (77, (E4M3_ONE, 1.0)), (127, (E4M3_ONE, 1.0))]:
        inp = _blank_decode(1, page, npages, L, 1, 16, 4)
        inp.q[0, 0, dstar] = qcode
        inp.q_scale[0] = qscale
        expect = np.empty(L)
        for p in range(L):
            nib = (p * 7 + dstar) % 16
            sc = 118 + (p % 17)
            _set_key(inp, p, dstar, nib, sc)
            # a decoy in the other nibble of the same byte and in another group
            _set_key(inp, p, dstar ^ 1, 7, sc)
            _set_key(inp, p, (dstar + 32) % 128, 7, 127 + (p % 3))
            expect[p] = max(0.0, _e2m1(nib) * 2.0 ** (sc - 127))
        got = orc.logits_paged(inp, 0, 0, L)
        assert np.array_equal(got, expect), \
            f"one-hot d*={dstar}: first mismatch at {int(np.flatnonzero(got != expect)[0])}"


def pin_relu_sign(orc):
    """Two heads, w = (1, -1/2): L[p] = max(0, a_p) - max(0, b_p)/2."""
    page, npages, L = 16, 4, 64
    inp = _blank_decode(2, page, npages, L, 1, 16, 4)
    inp.weights[0] = [BF16_ONE, 0xBF00]  # 1.0, -0.5
    inp.q[0, 0, 5] = E4M3_ONE
    inp.q[0, 1, 70] = E4M3_ONE
    expect = np.empty(L)
    for p in range(L):
        na, nb = p % 16, (3 * p + 1) % 16
        _set_key(inp, p, 5, na, 127)
        _set_key(inp, p, 70, nb, 126)
        a, b = _e2m1(na), _e2m1(nb) * 0.5
        expect[p] = max(0.0, a) - 0.5 * max(0.0, b)
    got = orc.logits_paged(inp, 0, 0, L)
    assert np.array_equal(got, expect), "relu/sign closed form"


def _bitfield_e4m3(c):
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def _bitfield_bf16(b):
    s, e, m = b >> 15, (b >> 7) & 255, b & 127
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def pin_exact_rational(orc):
    """Random tiny decode row, H=2: the oracle's double result equals the
    exact rational value to within a few ulps."""
    rng = np.random.Generator(np.random.PCG64(11))
    h, page, npages, L = 2, 16, 4, 64
    inp = _blank_decode(h, page, npages, L, 1, 16, 4)
    x = rng.standard_normal((1, h, 128)).astype(np.float32)
    inp.q, inp.q_scale = synth.quantize_q(x)
    inp.weights[0] = synth.encode_bf16(rng.standard_normal(h).astype(np.float32))
    v, s = synth.quantize_k_tokens(rng.standard_normal((npages * page, 128)).astype(np.float32))
    synth.write_pages(inp.k_cache, np.arange(npages), v, s, page)
    got = orc.logits_paged(inp, 0, 0, L)
    qs = Fraction(float(inp.q_scale[0]))
    for p in range(L):
        page_id = int(inp.block_table[0][p // page])
        tok = p % page
        vals = inp.k_cache[page_id, tok * 64:(tok + 1) * 64]
        scl = inp.k_cache[page_id, page * 64 + tok * 4: page * 64 + tok * 4 + 4]
        k = []
        for d in range(128):
            nib = (int(vals[d // 2]) >> (4 * (d % 2))) & 15
            k.append(Fraction(_e2m1(nib)) * Fraction(2) ** (int(scl[d // 32]) - 127))
        exact = Fraction(0)
        for hh in range(h):
            dot = sum(_bitfield_e4m3(int(inp.q[0, hh, d])) * qs * k[d] for d in range(128))
            exact += _bitfield_bf16(int(inp.weights[0, hh])) * max(Fraction(0), dot)
        assert abs(Fraction(got[p]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200), \
            f"exact rational mismatch at {p}: {got[p]} vs {float(exact)}"


def _np_tables():
    e4m3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()
    e2m1 = np.array([_e2m1(c) for c in range(16)])
    return e4m3, e2m1


def _np_keys_paged(inp, req, L):
    """[L, D] float64 keys of one request by numpy indexing."""
    g = inp.geom
    e4m3, e2m1 = _np_tables()
    p = np.arange(L)
    pages = inp.block_table[req][p // g.page_size].astype(np.int64)
    tok = p % g.page_size
    vals = inp.k_cache[pages[:, None], tok[:, None] * 64 + np.arange(64)[None, :]]
    scl = inp.k_cache[pages[:, None], g.page_size * 64 + tok[:, None] * 4 + np.arange(4)[None, :]]
    nib = np.stack([vals & 15, vals >> 4], axis=2).reshape(L, 128)
    return e2m1[nib] * np.ldexp(1.0, np.repeat(scl.astype(np.int64) - 127, 32, axis=1))


def _np_logits(q8, qs, w16, keys):
    e4m3, _ = _np_tables()
    q = e4m3[q8] * float(qs)
    w = (w16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dots = np.einsum("hd,pd->hp", q, keys)
    return (np.maximum(dots, 0.0) * w[:, None]).sum(axis=0)


def pin_numpy_einsum(orc):
    inp = synth.tiny_decode(0)
    for r in range(inp.rows):
        L = int(inp.row_ke[r])
        keys = _np_keys_paged(inp, int(inp.row_indices[r]), L)
        ref = _np_logits(inp.q[r], inp.q_scale[r], inp.weights[r], keys)
        got = orc.logits_paged(inp, r, 0, L)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12, err_msg=f"row {r}")
    # contiguous K (prefill): small two-sequence case
    pf = synth.prefill_chunk(seed=9, seq_lens=(300, 200), queries_per_seq=4, num_heads=16,
                             page_size=64, cbs=64, ncb=2, topk=16)
    kv, kscl = oracle_pkg.gather_reference(pf, orc)
    e4m3, e2m1 = _np_tables()
    nib = np.stack([kv & 15, kv >> 4], axis=2).reshape(kv.shape[0], 128)
    keys_all = e2m1[nib] * np.ldexp(1.0, np.repeat(kscl.astype(np.int64) - 127, 32, axis=1))
    for r in range(pf.rows):
        ks, ke = int(pf.cu_seqlen_ks[r]), int(pf.cu_seqlen_ke[r])
        ref = _np_logits(pf.q[r], pf.q_scale[r], pf.weights[r], keys_all[ks:ke])
        got = orc.logits_contig(pf, kv, kscl, r, 0, ke - ks)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12, err_msg=f"prefill row {r}")


def _monotone_input(L, cand, topk, cbs=16, page=16, npages=12):
    """K[p, 0:32] all equal to (1 or 1.5) * 2^e with e growing every two
    positions, so K[p, 0] = 1, 1.5, 2, 3, 4, 6, ... times 2^-27; q = 1 on
    d in [0, 32) => logits strictly increasing in p."""
    inp = _blank_decode(1, page, npages, L, len(cand), cbs, topk)
    inp.candidate_blocks[0] = cand
    inp.q[0, 0, :32] = E4M3_ONE
    for p in range(L):
        nib, sc = 2 + (p % 2), 100 + p // 2
        for d in range(32):
            _set_key(inp, p, d, nib, sc)
    return inp


def pin_monotone_topk(orc):
    cbs = 16
    cand = np.array([3, -1, 0, 3, 9, 5, 40, -7], dtype=np.int32)  # repeats, -1, <-1, out of range
    L = 150
    for topk in (5, 40, 64, 200):
        inp = _monotone_input(L, cand, topk)
        res = oracle_pkg.reference_rows(inp, [0], mode="dense", threads=1, orc=orc)[0]
        valid = sorted({b * cbs + j for b in cand if b >= 0 for j in range(cbs) if b * cbs + j < L})
        want = list(reversed(valid))[:topk]
        want += [-1] * (topk - len(want))
        assert res.topk.tolist() == want, f"monotone top-{topk}: {res.topk.tolist()[:10]} vs {want[:10]}"
        assert np.array_equal(np.flatnonzero(res.valid), valid), "candidate mask"


def pin_ties(orc):
    """Every key equal -> every valid logit equal -> the k smallest positions."""
    cbs, L, topk = 16, 150, 20
    cand = np.array([7, 2, 4, -1], dtype=np.int32)
    inp = _blank_decode(1, 16, 12, L, len(cand), cbs, topk)
    inp.candidate_blocks[0] = cand
    inp.q[0, 0, :] = E4M3_ONE
    for p in range(L):
        for d in range(0, 128, 9):
            _set_key(inp, p, d, 3, 127)
    res = oracle_pkg.reference_rows(inp, [0], mode="dense", threads=1, orc=orc)[0]
    valid = sorted(b * cbs + j for b in cand if b >= 0 for j in range(cbs) if b * cbs + j < L)
    assert res.topk.tolist() == valid[:topk], "ties go to the lower position"
    vals = res.logits[valid]
    assert np.all(vals == vals[0]) and vals[0] > 0


def pin_padding(orc):
    """Tiny row 3 has 40 valid positions and k = 64: 40 ids then 24 x -1."""
    inp = synth.tiny_decode(0)
    res = oracle_pkg.reference_rows(inp, [3], mode="dense", threads=1, orc=orc)[3]
    assert res.end == 40
    assert np.all(res.topk[:40] >= 0) and np.all(res.topk[40:] == -1)
    assert sorted(res.topk[:40].tolist()) == list(range(40))
    # an empty row: every id -1
    inp.row_ke[3] = 0
    res = oracle_pkg.reference_rows(inp, [3], mode="dense", threads=1, orc=orc)[3]
    assert res.end == 0 and np.all(res.topk == -1)


def pin_expansion_golden(orc):
    with open(os.path.join(GOLDEN, "expansion_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        si, end = orc.expand(c["cbs"], c["sbkv"], np.array(c["cand"], np.int32), c["L"], c["nsb"])
        assert si.tolist() == c["sparse_indices"], f"{c['name']}: {si.tolist()}"
        assert end == c["end"], f"{c['name']}: end {end} != {c['end']}"


def pin_gather(orc):
    pf = synth.prefill_chunk(seed=9, seq_lens=(300, 200), queries_per_seq=4, num_heads=16,
                             page_size=64, cbs=64, ncb=2, topk=16)
    kv, ks = oracle_pkg.gather_reference(pf, orc)
    g = pf.geom
    for s in range(2):
        a, b = int(pf.cu_seq_lens[s]), int(pf.cu_seq_lens[s + 1])
        for p in range(b - a):
            page = int(pf.seq_block_table[s][p // g.page_size])
            tok = p % g.page_size
            assert np.array_equal(kv[a + p], pf.k_cache[page, tok * 64:(tok + 1) * 64])
            off = g.page_size * 64 + tok * 4
            assert np.array_equal(ks[a + p], pf.k_cache[page, off:off + 4])


def pin_dense_equals_sparse(orc):
    """The candidate-only result equals the dense-then-masked result."""
    inp = synth.tiny_decode(0)
    dense = oracle_pkg.reference_rows(inp, mode="dense", threads=2, orc=orc)
    sparse = oracle_pkg.reference_rows(inp, mode="sparse", threads=2, orc=orc)
    for r in range(inp.rows):
        d, s = dense[r], sparse[r]
        assert np.array_equal(np.flatnonzero(d.valid), np.sort(s.positions)), f"row {r}: columns"
        assert np.array_equal(d.logits[s.positions], s.logits), f"row {r}: logits"
        assert np.array_equal(d.topk, s.topk), f"row {r}: top-k"


ALL_PINS = [
    pin_e4m3, pin_bf16, pin_e2m1, pin_ue8m0, pin_one_hot, pin_relu_sign, pin_exact_rational,
    pin_numpy_einsum, pin_monotone_topk, pin_ties, pin_padding, pin_expansion_golden, pin_gather,
    pin_dense_equals_sparse,
]
