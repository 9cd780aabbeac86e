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
  encoders                 E2M1: the OCP table's values and midpoints (ties to
                           the even code), saturation; E4M3 and bf16 against
                           torch's float8_e4m3fn / bfloat16 casts (nearest even)
  k_scale_cases            hand-worked scale exponents: amax at and past
                           6 * 2^e, zeros, the clamp at the smallest code
  k_nearest                brute force: each decoded element is the nearest
                           point of its group's grid, the exponent is the
                           smallest that covers the group's amax
  k_cache_layout           numpy slicing: each token's bytes sit at its slot's
                           page and offset; other bytes stay untouched; a
                           one-hot query reads the written keys back
  q_quantiser              torch: scale = amax / 448 in float32, codes of
                           x / scale cast to float8_e4m3fn, bf16 weights
  source_hand              candidate source, hand-worked: block maxima set
                           through the one-hot closed form, a tie, a partial
                           last block, a block of zeros, -1 padding
  source_monotone_ties     increasing keys -> the last blocks first; equal
                           keys -> the first blocks
  source_numpy             random logits: numpy block maxima (padded with
                           -inf) and a lexsort on (-max, block id)
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


# -------------------------------------------------------------- producers


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def pin_encoders(orc):
    for c in range(16):  # every table value to its own code (zero keeps its sign)
        v = -0.0 if c == 8 else _e2m1(c)
        assert orc.encode_e2m1(v) == c, f"e2m1 encode of {v}: {orc.encode_e2m1(v)} != {c}"
    for i in range(7):  # midpoints to the even code of the two neighbours
        mid = (E2M1_TABLE[i] + E2M1_TABLE[i + 1]) / 2
        want = i if i % 2 == 0 else i + 1
        assert orc.encode_e2m1(mid) == want, f"e2m1 midpoint {mid}"
        assert orc.encode_e2m1(-mid) == want | 8, f"e2m1 midpoint {-mid}"
        assert orc.encode_e2m1(mid * 0.999) == i and orc.encode_e2m1(mid * 1.001) == i + 1
    assert orc.encode_e2m1(6.5) == 7 and orc.encode_e2m1(1e30) == 7 and orc.encode_e2m1(-7.0) == 15
    # E4M3 against torch: every finite value, every midpoint between neighbours, random values
    vals = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.Generator(np.random.PCG64(17))
    xs = np.concatenate([vals, -vals, mids, -mids, rng.uniform(-450, 450, 3000), rng.normal(0, 1, 3000)])
    xs = xs.astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert orc.encode_e4m3(x) == r, f"e4m3 encode of {x!r}: {orc.encode_e4m3(x):#x} != {r:#x}"
    assert orc.encode_e4m3(1e6) == 0x7E and orc.encode_e4m3(-1e6) == 0xFE
    # bf16 against torch: ties between neighbours and random floats
    fs = np.concatenate([1.0 + np.arange(1, 64) * 2.0 ** -8, rng.normal(0, 3, 4000)]).astype(np.float32)
    ref = _bf16_bits(fs)
    for f, r in zip(fs.tolist(), ref.tolist()):
        assert orc.encode_bf16(f) == r, f"bf16 encode of {f!r}"


def _token(values):
    k = np.zeros(128, dtype=np.float32)
    k[:len(values)] = values
    return _bf16_bits(k)


def pin_k_scale_cases(orc):
    # (group 0's values, expected UE8M0 code): the smallest e with amax <= 6 * 2^e
    cases = [([6.0], 127), ([6.03125], 128), ([-3.0], 126), ([3.015625, 1.0], 127), ([0.75], 124),
             ([12.0], 128), ([12.0625], 129), ([1.0], 125), ([2.0 ** -130], 1), ([0.0], 127)]
    for vals, code in cases:
        v, sc = orc.quantize_k_token(_token(vals))
        assert sc[0] == code, f"scale of amax {max(abs(x) for x in vals)}: {sc[0]} != {code}"
        assert sc[1:].tolist() == [127, 127, 127], "groups of zeros take code 127"
    v, sc = orc.quantize_k_token(_token([6.0, -3.0, 0.25, 0.75]))  # scale 1: codes 7, 13 (-3), 0, 2
    assert v[0] == (7 | (13 << 4)) and v[1] == (0 | (2 << 4)), f"packed codes {v[:2]}"
    v, sc = orc.quantize_k_token(_token([0.0] * 32 + [-0.5]))  # group 1, element 32: low nibble of byte 16
    assert v[16] == 14 and sc[1] == 124, f"group 1 element {v[16]}, scale {sc[1]}"  # -0.5 = -4 * 2^-3


def pin_k_nearest(orc):
    rng = np.random.Generator(np.random.PCG64(23))
    grid = np.array(sorted({s * t for t in E2M1_TABLE for s in (-1.0, 1.0)}))
    for trial in range(40):
        scale = 2.0 ** rng.integers(-20, 20)
        x = (rng.standard_normal(128) * scale * (1 + 3 * (trial % 3))).astype(np.float32)
        kb = _bf16_bits(x)
        xv = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        v, sc = orc.quantize_k_token(kb)
        for g in range(4):
            e = int(sc[g]) - 127
            seg = xv[32 * g:32 * g + 32]
            amax = np.abs(seg).max()
            assert amax <= 6 * 2.0 ** e and (amax > 6 * 2.0 ** (e - 1) or sc[g] == 1), f"group {g} exponent"
            for i in range(32):
                d = 32 * g + i
                code = (v[d // 2] >> (4 * (d % 2))) & 15
                got = _e2m1(code) * 2.0 ** e
                best = np.abs(grid * 2.0 ** e - seg[i]).min()
                assert abs(got - seg[i]) == best, f"element {d}: {got} is not a nearest grid point of {seg[i]}"


def pin_k_cache_layout(orc):
    rng = np.random.Generator(np.random.PCG64(29))
    page, npages, ntok = 16, 6, 40
    pb = page * 68
    k = _bf16_bits(rng.standard_normal((ntok, 128)).astype(np.float32))
    slots = rng.permutation(page * npages)[:ntok].astype(np.int64)
    slots[::7] = -1
    cache = np.full((npages, pb), 0xA5, dtype=np.uint8)
    orc.write_k_cache(k, slots, cache, page)
    expect = np.full((npages, pb), 0xA5, dtype=np.uint8)
    for t in range(ntok):
        if slots[t] < 0:
            continue
        pg, off = divmod(int(slots[t]), page)
        v, sc = orc.quantize_k_token(k[t])
        expect[pg, off * 64:(off + 1) * 64] = v
        expect[pg, page * 64 + off * 4:page * 64 + (off + 1) * 4] = sc
    assert np.array_equal(cache, expect), "written page bytes"
    # read back through the decode path: a one-hot query at d* gives max(0, K[t, d*])
    g = synth.Geometry(8, 128, page, 16, 1, 1)
    bt = np.arange(npages, dtype=np.int32)[None, :]
    for d in (0, 33, 127):
        q8 = np.zeros((1, 8, 128), dtype=np.uint8)
        q8[0, 0, d] = E4M3_ONE
        w = np.zeros((1, 8), dtype=np.uint16)
        w[0, 0] = BF16_ONE
        inp = synth.DecodeInputs(g, q8, np.array([1.0], dtype=np.float32), w, cache, bt,
                                 np.zeros(1, dtype=np.int32), np.array([page * npages], dtype=np.int32),
                                 np.zeros((1, 1), dtype=np.int32))
        logits = orc.logits_paged(inp, 0, 0, page * npages)
        for t in range(ntok):
            if slots[t] < 0:
                continue
            v, sc = orc.quantize_k_token(k[t])
            kd = _e2m1((v[d // 2] >> (4 * (d % 2))) & 15) * 2.0 ** (int(sc[d // 32]) - 127)
            assert abs(logits[slots[t]] - max(0.0, kd)) <= 1e-12 * max(1.0, abs(kd)), f"token {t} d {d}"


def pin_q_quantiser(orc):
    rng = np.random.Generator(np.random.PCG64(31))
    R, H = 5, 16
    x = rng.standard_normal((R, H, 128)).astype(np.float32) * np.array([1, 1e-3, 40, 1, 2], dtype=np.float32)[:, None, None]
    x[3] = 0.0  # a zero row: scale 1
    qb = _bf16_bits(x)
    w = rng.standard_normal((R, H)).astype(np.float32)
    q8, sc, wb = orc.quantize_q(qb, w)
    xt = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    amax = xt.abs().reshape(R, -1).amax(dim=1)
    st = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert np.array_equal(sc, st.numpy()), "per-row scale amax / 448"
    ref = (xt / st[:, None, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q8, ref), "E4M3 codes of x / scale"
    assert np.array_equal(wb, _bf16_bits(w)), "bf16 weights"


# -------------------------------------------------------------- candidate source


def pin_source_hand(orc):
    """One head, one-hot query at d = 5: L[p] = max(0, K[p, 5]). cbs = 16,
    L = 75 (five blocks, the last of 11 positions). Block maxima by hand:
    1.0, 3.0, 0, 3.0, 6.0 -> blocks 4, 1, 3 (tie with 1, higher id), 0, 2, then -1."""
    inp = _blank_decode(8, 16, 6, 75, 7, 16, 4)
    inp.q[0, 0, 5] = E4M3_ONE
    inp.weights[0, 1:] = 0
    # (position, E2M1 code): 1.0 = code 2, 3.0 = code 5, 6.0 = code 7, 0.5 = code 1, -6 = code 15
    for p, code in [(3, 2), (7, 1), (20, 5), (31, 2), (40, 15), (50, 5), (49, 1), (74, 7), (66, 5)]:
        _set_key(inp, p, 5, code, 127)
    cand, scores, logits = orc_source_row(orc, inp)
    assert scores.tolist() == [1.0, 3.0, 0.0, 3.0, 6.0], f"block maxima {scores.tolist()}"
    assert cand.tolist() == [4, 1, 3, 0, 2, -1, -1], f"published blocks {cand.tolist()}"


def orc_source_row(orc, inp):
    return oracle_pkg.source_rows(inp, rows=[0], orc=orc)[0]


def pin_source_monotone_ties(orc):
    inp = _monotone_input(90, [-1] * 4, 8)  # cbs 16: blocks 0..5, the last of 10 positions
    inp.geom = synth.Geometry(1, 128, 16, 16, 4, 8)
    cand, scores, logits = orc_source_row(orc, inp)
    assert cand.tolist() == [5, 4, 3, 2], f"increasing keys: {cand.tolist()}"
    flat = _blank_decode(8, 16, 6, 64, 6, 16, 4)  # every key zero: every logit 0, every block ties
    cand, scores, logits = orc_source_row(orc, flat)
    assert cand.tolist() == [0, 1, 2, 3, -1, -1], f"equal keys: {cand.tolist()}"


def pin_source_numpy(orc):
    rng = np.random.Generator(np.random.PCG64(37))
    for L, cbs, ncb in [(1000, 64, 8), (97, 16, 10), (5, 16, 3), (4096, 128, 32), (130, 128, 4)]:
        logits = np.round(rng.standard_normal(L), 1)  # rounding makes block-maximum ties
        cand, scores = orc.source_blocks(logits, cbs, ncb)
        nb = -(-L // cbs)
        padded = np.full(nb * cbs, -np.inf)
        padded[:L] = logits
        mx = padded.reshape(nb, cbs).max(axis=1)
        assert np.array_equal(scores, mx), f"block maxima L={L}"
        order = np.lexsort((np.arange(nb), -mx))[:ncb]
        want = np.full(ncb, -1)
        want[:len(order)] = order
        assert np.array_equal(cand, want), f"published blocks L={L}: {cand.tolist()} != {want.tolist()}"


ALL_PINS = [
    pin_e4m3, pin_bf16, pin_e2m1, pin_ue8m0, pin_one_hot, pin_relu_sign, pin_exact_rational,
    pin_numpy_einsum, pin_monotone_topk, pin_ties, pin_padding, pin_expansion_golden, pin_gather,
    pin_dense_equals_sparse, pin_encoders, pin_k_scale_cases, pin_k_nearest, pin_k_cache_layout, pin_q_quantiser,
    pin_source_hand, pin_source_monotone_ties, pin_source_numpy,
]
