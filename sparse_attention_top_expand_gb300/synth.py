"""Seeded synthetic inputs for the candidate-block sparse MQA-logits indexer.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path: it draws random tensors and ENCODES them into the byte formats the
indexer consumes (FP8 E4M3 queries with a per-row scale, MXFP4 keys in a
paged cache, bf16 head weights, block tables and candidate blocks).  It
holds none of the scoring arithmetic: nothing here decodes a code, takes a
dot product, applies ReLU, reduces over heads, masks or selects.

Formats written here (the byte layout is ours; the pages fix the element
formats only):

* Q: ``[rows, H, D]`` uint8 OCP FP8 E4M3 ("fn": max 448, no infinities),
  ``q_scale``: ``[rows]`` float32, one scale per query row (vLLM
  sparse_mqa_indexer docs, ``SparseMQAIndexer.forward``: ``q_quant`` is a
  ``(values, scales)`` pair and the decode call unsqueezes a per-row scale).
* weights: ``[rows, H]`` uint16 holding bfloat16 bits (same page,
  ``weights_dtype``).
* K cache page (``page_bytes = page_size * (D/2 + D/32)``): first the values
  ``[page_size][D/2]`` with element ``2i`` in the low nibble of byte ``i`` and
  ``2i+1`` in the high nibble, OCP MX FP4 E2M1; then the scales
  ``[page_size][D/32]``, byte ``g`` the UE8M0 exponent of elements
  ``[32g, 32g+32)`` (sparse_indexer.py, builder ``__init__``: the MXFP4
  indexer cache with UE8M0-packed granularity-32 scales).

Quantisers (generator only; both sides read the same bytes):

* E4M3: ``scale = amax/448`` in float32 (``amax == 0`` gives 1), value
  ``x/scale`` clamped to +-448 and rounded to nearest, ties to even code.
* MXFP4: per 32-group ``e = ceil(log2(amax/6))`` found exactly, code
  ``e + 127`` clamped to ``[1, 254]``; elements ``x * 2^-e`` rounded to the
  nearest E2M1 value (ties to even code), clamped to +-6.  ``amax == 0`` gives
  code 127 and zeros.
* bf16: round to nearest even from float32.

Random draws use numpy's PCG64 generator seeded per workload.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 128

# --------------------------------------------------------------------------
# Encoders (value -> code).  These are the quantisers of the generator.
# --------------------------------------------------------------------------

_E4M3_POS_CODES = np.arange(0, 127, dtype=np.int64)  # 0x00..0x7E, 0x7F is NaN
_e = _E4M3_POS_CODES >> 3
_m = _E4M3_POS_CODES & 7
_E4M3_POS_VALUES = np.where(_e == 0, (_m / 8.0) * 2.0 ** -6,
                            (1.0 + _m / 8.0) * np.exp2(_e - 7.0))
_E2M1_POS_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _round_to_table(a: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of an increasing table, ties to the even
    index (the even code).  ``a`` must be within [table[0], table[-1]]."""
    hi = np.searchsorted(table, a, side="left")
    hi = np.clip(hi, 1, len(table) - 1)
    lo = hi - 1
    dlo = a - table[lo]
    dhi = table[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float -> OCP FP8 E4M3 code, saturating at +-448, nearest-even."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    code = _round_to_table(a, _E4M3_POS_VALUES).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """float -> E2M1 nibble (0..15), saturating at +-6, nearest-even."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    code = _round_to_table(a, _E2M1_POS_VALUES).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(8), code).astype(np.uint8)


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def quantize_q(x: np.ndarray):
    """[rows, H, D] float32 -> (E4M3 codes [rows, H, D], float32 scale [rows])."""
    rows = x.shape[0]
    amax = np.abs(x.reshape(rows, -1)).max(axis=1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = encode_e4m3(x.astype(np.float64) / scale.astype(np.float64)[:, None, None])
    return codes, scale


def _group_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with amax <= 6 * 2^e (exact), per group."""
    safe = np.where(amax > 0, amax, 1.0)
    e = np.ceil(np.log2(safe / 6.0)).astype(np.int64)
    # log2 may be off by one near powers of two; settle it with exact tests.
    e = np.where(safe > 6.0 * np.exp2(e.astype(np.float64)), e + 1, e)
    e = np.where(safe <= 6.0 * np.exp2((e - 1).astype(np.float64)), e - 1, e)
    return e


def quantize_k_tokens(x: np.ndarray):
    """[ntok, D] float32 -> (packed values [ntok, D/2] uint8, scales [ntok, D/32] uint8)."""
    ntok, d = x.shape
    g = x.astype(np.float64).reshape(ntok, d // 32, 32)
    amax = np.abs(g).max(axis=2)
    e = _group_exponent(amax)
    code = np.clip(e + 127, 1, 254)
    e = code - 127
    e = np.where(amax > 0, e, 0)
    code = np.where(amax > 0, code, 127).astype(np.uint8)
    nib = encode_e2m1(g * np.exp2(-e.astype(np.float64))[:, :, None]).reshape(ntok, d)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return packed, code


def page_bytes(page_size: int, head_dim: int = HEAD_DIM) -> int:
    return page_size * (head_dim // 2 + head_dim // 32)


def write_pages(cache: np.ndarray, pages: np.ndarray, values: np.ndarray,
                scales: np.ndarray, page_size: int, head_dim: int = HEAD_DIM) -> None:
    """Store whole pages: values [len(pages)*page_size, D/2], scales [.., D/32]."""
    vb = page_size * head_dim // 2
    v = values.reshape(len(pages), vb)
    s = scales.reshape(len(pages), page_size * head_dim // 32)
    cache[pages, :vb] = v
    cache[pages, vb:] = s


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------


@dataclasses.dataclass
class Geometry:
    num_heads: int
    head_dim: int
    page_size: int
    candidate_block_size: int
    candidate_topk_blocks: int
    topk: int


@dataclasses.dataclass
class DecodeInputs:
    """One decode step: every row is one query token of one request."""

    geom: Geometry
    q: np.ndarray              # [R, H, D] uint8 E4M3
    q_scale: np.ndarray        # [R] float32
    weights: np.ndarray        # [R, H] uint16 bf16 bits
    k_cache: np.ndarray        # [num_pages, page_bytes] uint8
    block_table: np.ndarray    # [bt_rows, bt_cols] int32 (-1 = unused)
    row_indices: np.ndarray    # [R] int32, row -> block-table row
    row_ke: np.ndarray         # [R] int32 compressed context length
    candidate_blocks: np.ndarray  # [R, ncb] int32, units of cbs, -1 = none

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])


@dataclasses.dataclass
class PrefillInputs:
    """One prefill chunk: query rows of several sequences, K in a paged cache
    that the gather copies into a contiguous workspace."""

    geom: Geometry
    q: np.ndarray
    q_scale: np.ndarray
    weights: np.ndarray
    k_cache: np.ndarray            # paged cache the gather reads
    seq_block_table: np.ndarray    # [nseq, bt_cols] int32
    cu_seq_lens: np.ndarray        # [nseq+1] int32, offsets in the workspace
    cu_seqlen_ks: np.ndarray       # [R] int32, row K range start (workspace)
    cu_seqlen_ke: np.ndarray       # [R] int32, row K range end (exclusive)
    candidate_blocks: np.ndarray   # [R, ncb] int32, relative to ks

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def total_len(self) -> int:
        return int(self.cu_seq_lens[-1])


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _queries(rng, rows, h, d):
    x = rng.standard_normal((rows, h, d), dtype=np.float32)
    q, qs = quantize_q(x)
    w = rng.standard_normal((rows, h), dtype=np.float32) * np.float32(1.0 / math.sqrt(h))
    return q, qs, encode_bf16(w)


def _fill_cache(rng, num_pages, page_size, d, touched: np.ndarray):
    """N(0,1) MXFP4 keys on touched pages; random E2M1 codes with unit scale
    on pages no candidate block reaches (they never influence a result)."""
    pb = page_bytes(page_size, d)
    cache = np.empty((num_pages, pb), dtype=np.uint8)
    vb = page_size * d // 2
    untouched = np.setdiff1d(np.arange(num_pages), touched)
    if len(untouched):
        cache[untouched, :vb] = rng.integers(0, 256, size=(len(untouched), vb), dtype=np.uint8)
        cache[untouched, vb:] = 127
    touched = np.asarray(touched, dtype=np.int64)
    chunk = max(1, (1 << 22) // (page_size * d))  # pages per batch (~16 MB floats)
    for i in range(0, len(touched), chunk):
        pg = touched[i:i + chunk]
        x = rng.standard_normal((len(pg) * page_size, d), dtype=np.float32)
        v, s = quantize_k_tokens(x)
        write_pages(cache, pg, v, s, page_size, d)
    return cache


def _distinct_blocks(rng, nblk, ncb):
    """ncb distinct ids from [0, nblk); if fewer exist, all of them shuffled
    then -1 padding."""
    if nblk >= ncb:
        return rng.choice(nblk, size=ncb, replace=False).astype(np.int32)
    out = np.full(ncb, -1, dtype=np.int32)
    out[:nblk] = rng.permutation(nblk).astype(np.int32)
    return out


_I32_MIN, _I32_MAX = -(2 ** 31), 2 ** 31 - 1


def adversarial_blocks(rng, ncb, L, cbs, kind):
    """Candidate rows that exercise every rule of the expansion: ids repeated
    within the first 32 entries and between the first and second 32,
    -1 and other negative ids, blocks at and far past the row end.

    kind "mixed": a few distinct in-range ids, each repeated, among invalid
    ones; "lone": one in-range id repeated among invalid ones; "none": no
    in-range id at all."""
    nblk = (L + cbs - 1) // cbs
    invalid_pool = np.array([-1, -2, -7, -1000, _I32_MIN, nblk, nblk + 1, nblk + 5, 4 * nblk + 3,
                             _I32_MAX], dtype=np.int64)
    out = rng.choice(invalid_pool, size=ncb).astype(np.int64)
    if kind == "none" or nblk == 0:
        return out.astype(np.int32)
    if kind == "lone":
        b = int(rng.integers(0, nblk))
        slots = rng.choice(ncb, size=min(ncb, 3), replace=False)
        if ncb > 32:  # one copy in each half
            slots[0] = int(rng.integers(0, 32))
            slots[-1] = int(rng.integers(32, ncb))
        out[slots] = b
        return out.astype(np.int32)
    nd = max(1, min(nblk, ncb // 3))
    ids = rng.choice(nblk, size=nd, replace=False)
    # every distinct id once in a random slot, then repeats: some inside the
    # first 32 slots, some in the second 32 naming an id of the first
    slots = rng.permutation(ncb)
    out[slots[:nd]] = ids
    nrep = min(ncb - nd, nd)
    for j in range(nrep):
        out[slots[nd + j]] = ids[j % nd]
    if ncb > 32:
        lo = [s for s in range(32) if out[s] >= 0 and out[s] < nblk]
        if lo:
            out[int(rng.integers(32, ncb))] = out[lo[0]]
    return out.astype(np.int32)


def _touched_pages(block_table, row_indices, row_ke, cand, cbs, page_size):
    pages = set()
    for r in range(cand.shape[0]):
        bt = block_table[row_indices[r]]
        L = int(row_ke[r])
        for b in cand[r]:
            b = int(b)
            if b < 0 or b * cbs >= L:
                continue
            for p in range(b * cbs, min((b + 1) * cbs, L), page_size):
                pages.add(int(bt[p // page_size]))
    return np.array(sorted(pages), dtype=np.int64)


def _paged_decode(seed, rows, h, page_size, cbs, ncb, topk, ctx, cand_fn=None,
                  row_perm=False, shared_pool_pages: Optional[int] = None):
    d = HEAD_DIM
    rng = _rng(seed)
    geom = Geometry(h, d, page_size, cbs, ncb, topk)
    q, qs, w = _queries(rng, rows, h, d)
    npages_req = [(int(c) + page_size - 1) // page_size for c in ctx]
    bt_cols = max(npages_req)
    if shared_pool_pages is not None:
        num_pages = shared_pool_pages
        bt = np.stack([rng.permutation(num_pages)[:bt_cols] for _ in range(rows)]).astype(np.int32)
    else:
        num_pages = int(sum(npages_req))
        perm = rng.permutation(num_pages).astype(np.int32)
        bt = np.full((rows, bt_cols), -1, dtype=np.int32)
        off = 0
        for j, n in enumerate(npages_req):
            bt[j, :n] = perm[off:off + n]
            off += n
    row_indices = (rng.permutation(rows) if row_perm else np.arange(rows)).astype(np.int32)
    row_ke = np.asarray(ctx, dtype=np.int32)[row_indices]
    cand = np.empty((rows, ncb), dtype=np.int32)
    for r in range(rows):
        L = int(row_ke[r])
        if cand_fn is not None:
            cand[r] = cand_fn(rng, r, L)
        else:
            cand[r] = _distinct_blocks(rng, (L + cbs - 1) // cbs, ncb)
    touched = _touched_pages(bt, row_indices, row_ke, cand, cbs, page_size)
    cache = _fill_cache(rng, num_pages, page_size, d, touched)
    return DecodeInputs(geom, q, qs, w, cache, bt, row_indices, row_ke, cand)


def tiny_decode(seed: int = 0) -> DecodeInputs:
    """4 decode rows, H=8, one 1024-position pool in 16 pages of 64 that every
    row maps through its own permuted block table; cbs=64, 4 blocks per row,
    topk=64.  Row 2 has a -1 block; row 3 has 40 positions (< topk) and only
    block 0 of its four is in range; rows map to block-table rows through a
    non-identity permutation."""
    rows, h, d, page, cbs, ncb, topk, pool = 4, 8, HEAD_DIM, 64, 64, 4, 64, 16
    rng = _rng(seed)
    geom = Geometry(h, d, page, cbs, ncb, topk)
    q, qs, w = _queries(rng, rows, h, d)
    bt = np.stack([rng.permutation(pool) for _ in range(rows)]).astype(np.int32)
    row_indices = np.array([2, 0, 3, 1], dtype=np.int32)
    row_ke = np.array([1024, 1024, 1024, 40], dtype=np.int32)
    cand = np.empty((rows, ncb), dtype=np.int32)
    cand[0] = rng.choice(pool, size=ncb, replace=False)
    cand[1] = rng.choice(pool, size=ncb, replace=False)
    c2 = np.concatenate([rng.choice(pool, size=3, replace=False), [-1]])
    cand[2] = rng.permutation(c2)
    c3 = np.concatenate([[0], rng.choice(np.arange(1, pool), size=3, replace=False)])
    cand[3] = rng.permutation(c3)
    cache = _fill_cache(rng, pool, page, d, np.arange(pool))
    return DecodeInputs(geom, q, qs, w, cache, bt, row_indices, row_ke, cand)


def decode_batch(seed: int = 1, rows: int = 64) -> DecodeInputs:
    """64 rows, H=64, contexts uniform in [4096, 32768], cbs=128 with 32
    distinct in-range blocks per row, page 64, topk=2048."""
    rng = _rng(seed + 7)
    ctx = rng.integers(4096, 32768 + 1, size=rows)
    return _paged_decode(seed, rows, 64, 64, 128, 32, 2048, ctx, row_perm=False)


def multi_token_decode(seed: int = 5, requests: int = 32, next_n: int = 2, num_heads: int = 64,
                       page_size: int = 64, cbs: int = 128, ncb: int = 32, topk: int = 2048,
                       ctx_range=(4096, 32768)) -> DecodeInputs:
    """Decode with next_n query tokens per request (speculative decoding): rows
    are request-major, row r is token r % next_n of request r // next_n, maps
    to that request's block-table row through row_indices, and sees its causal
    context: the request's length minus next_n, plus the token's index plus
    one. Each row has its own ncb distinct candidate blocks below its end."""
    d = HEAD_DIM
    rng = _rng(seed)
    geom = Geometry(num_heads, d, page_size, cbs, ncb, topk)
    rows = requests * next_n
    q, qs, w = _queries(rng, rows, num_heads, d)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=requests)
    npages_req = [(int(c) + page_size - 1) // page_size for c in ctx]
    num_pages = int(sum(npages_req))
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((requests, max(npages_req)), -1, dtype=np.int32)
    off = 0
    for j, n in enumerate(npages_req):
        bt[j, :n] = perm[off:off + n]
        off += n
    row_indices = (np.arange(rows) // next_n).astype(np.int32)
    row_ke = np.array([int(ctx[r // next_n]) - next_n + (r % next_n) + 1 for r in range(rows)], dtype=np.int32)
    cand = np.empty((rows, ncb), dtype=np.int32)
    for r in range(rows):
        cand[r] = _distinct_blocks(rng, (int(row_ke[r]) + cbs - 1) // cbs, ncb)
    touched = _touched_pages(bt, row_indices, row_ke, cand, cbs, page_size)
    cache = _fill_cache(rng, num_pages, page_size, d, touched)
    return DecodeInputs(geom, q, qs, w, cache, bt, row_indices, row_ke, cand)


def long_context_decode(seed: int = 4, rows: int = 256) -> DecodeInputs:
    """256 rows, H=64, contexts log-uniform in [2048, 131072] with 10% of rows
    shorter than topk (uniform in [1, 2047]); cbs=128, 64 blocks per row
    (all valid blocks then -1 where fewer exist), page 64, topk=2048."""
    rng = _rng(seed + 7)
    ctx = np.floor(np.exp(rng.uniform(math.log(2048), math.log(131072), size=rows))).astype(np.int64)
    short = rng.choice(rows, size=max(1, rows // 10), replace=False)
    ctx[short] = rng.integers(1, 2048, size=len(short))
    return _paged_decode(seed, rows, 64, 64, 128, 64, 2048, ctx, row_perm=False)


def shared_schedule_layers(seed: int = 3, layers: int = 4, rows: int = 64):
    """The decode batch's rows, block tables and candidates, with each layer's
    own queries, weights and K cache."""
    base = decode_batch(seed=1, rows=rows)
    out = []
    for li in range(layers):
        rng = _rng(seed * 100 + li)
        g = base.geom
        q, qs, w = _queries(rng, rows, g.num_heads, g.head_dim)
        touched = _touched_pages(base.block_table, base.row_indices, base.row_ke,
                                 base.candidate_blocks, g.candidate_block_size, g.page_size)
        cache = _fill_cache(rng, base.k_cache.shape[0], g.page_size, g.head_dim, touched)
        out.append(DecodeInputs(g, q, qs, w, cache, base.block_table, base.row_indices,
                                base.row_ke, base.candidate_blocks))
    return out


def prefill_as_decode(inp: PrefillInputs) -> DecodeInputs:
    """The chunk's rows as paged decode rows, for in-place paged prefill (no
    gather): row r reads its sequence's pages through the sequence's
    block-table row, with its causal end, relative to the sequence start, as
    its context length. Candidate blocks and output ids stay relative to the
    sequence start. Every row's range must start at its sequence's start."""
    ks = np.asarray(inp.cu_seqlen_ks, dtype=np.int64)
    seq = np.searchsorted(np.asarray(inp.cu_seq_lens, dtype=np.int64), ks, side="right") - 1
    if not np.array_equal(np.asarray(inp.cu_seq_lens)[seq], ks):
        raise ValueError("a row's key range does not start at its sequence's start")
    return DecodeInputs(geom=inp.geom, q=inp.q, q_scale=inp.q_scale, weights=inp.weights, k_cache=inp.k_cache,
                        block_table=inp.seq_block_table, row_indices=seq.astype(np.int32),
                        row_ke=(np.asarray(inp.cu_seqlen_ke, dtype=np.int64) - ks).astype(np.int32),
                        candidate_blocks=inp.candidate_blocks)


def prefill_chunk(seed: int = 2, seq_lens=(28672, 36864), queries_per_seq: int = 2048,
                  num_heads: int = 64, page_size: int = 64, cbs: int = 128,
                  ncb: int = 32, topk: int = 2048, cand_fn=None) -> PrefillInputs:
    """Query rows are the last ``queries_per_seq`` compressed positions of each
    sequence; row t of a sequence of length L sees positions [0, L - n + t + 1)
    (causal).  Candidate blocks: ncb distinct ids below the row's end, or
    ``cand_fn(rng, row, n)`` when given."""
    d = HEAD_DIM
    rng = _rng(seed)
    geom = Geometry(num_heads, d, page_size, cbs, ncb, topk)
    nseq = len(seq_lens)
    rows = nseq * queries_per_seq
    q, qs, w = _queries(rng, rows, num_heads, d)
    npages = [(L + page_size - 1) // page_size for L in seq_lens]
    num_pages = int(sum(npages))
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((nseq, max(npages)), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(npages):
        bt[s, :n] = perm[off:off + n]
        off += n
    cu = np.zeros(nseq + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seq_lens)
    ks = np.empty(rows, dtype=np.int32)
    ke = np.empty(rows, dtype=np.int32)
    cand = np.empty((rows, ncb), dtype=np.int32)
    r = 0
    for s, L in enumerate(seq_lens):
        for t in range(queries_per_seq):
            n = L - queries_per_seq + t + 1
            ks[r] = cu[s]
            ke[r] = cu[s] + n
            if cand_fn is not None:
                cand[r] = cand_fn(rng, r, n)
            else:
                cand[r] = _distinct_blocks(rng, (n + cbs - 1) // cbs, ncb)
            r += 1
    cache = _fill_cache(rng, num_pages, page_size, d, np.arange(num_pages))
    return PrefillInputs(geom, q, qs, w, cache, bt, cu, ks, ke, cand)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "decode_batch": decode_batch,
    "prefill_chunk": prefill_chunk,
    "shared_schedule": shared_schedule_layers,
    "long_context_decode": long_context_decode,
    "multi_token_decode": multi_token_decode,
}
