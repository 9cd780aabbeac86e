"""CPU oracle for the candidate-block sparse MQA-logits top-k indexer.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package. The product path (the CUDA library and its Python binding) never
does, and it shares no code with this package: the oracle is plain C in
double precision (``smq_oracle.c``) plus the row bookkeeping below.

Parity status of each function (the pins live in ``tests/test_oracle_pins.py``):
  - e4m3, bf16 decoders: every code against torch's float8_e4m3fn / bfloat16
    casts.
  - e2m1, ue8m0 decoders: the OCP MX v1.0 value table, and 2^(e-127) through
    math.ldexp.
  - dense logits: a one-hot closed form (pins the nibble order, the group
    index and the page walk); exact rational arithmetic on tiny inputs; and
    numpy float64 einsum over independently decoded tensors.
  - candidate mask and top-k: the monotone closed form, the all-equal (ties)
    case and the -1 padding case.
  - expansion: hand-derived cases in ``tests/golden/expansion_cases.json``.
  - gather: numpy slicing of the page bytes.
  - dense-then-masked == candidate-only: an invariant checked on every small
    workload.
  - candidate source (block scores, published blocks): hand-worked maxima
    through the one-hot closed form; the monotone and all-equal keys;
    a short context; brute-force ranking by numpy.
  - producers (K-cache writer, query quantiser): E2M1 / E4M3 / bf16 encoders
    against the value tables' midpoints and torch's float8_e4m3fn / bfloat16
    casts; hand-worked scale exponents; nearest-grid-point brute force; the
    page layout through the oracle's own decode path.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Iterable, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "smq_oracle.c")
DEFAULT_LIB = os.path.join(_HERE, "_build", "libsmq_oracle.so")

_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(out_path: str = DEFAULT_LIB, source: str = SOURCE, defines: Iterable[str] = ()) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-I", _HERE]
    cmd += ["-D" + d for d in defines]
    cmd += [source, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, lib_path: Optional[str] = None):
        if lib_path is None:
            lib_path = DEFAULT_LIB
            if not os.path.exists(lib_path) or os.path.getmtime(lib_path) < os.path.getmtime(SOURCE):
                build(lib_path)
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        for name in ("smq_oracle_e4m3", "smq_oracle_e2m1", "smq_oracle_ue8m0"):
            f = getattr(lib, name)
            f.restype = ctypes.c_double
            f.argtypes = [ctypes.c_uint8]
        lib.smq_oracle_bf16.restype = ctypes.c_double
        lib.smq_oracle_bf16.argtypes = [ctypes.c_uint16]
        lib.smq_oracle_logits_paged.restype = ctypes.c_int
        lib.smq_oracle_logits_paged.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, ctypes.c_float, _u16p,
            _u8p, ctypes.c_int64, _i32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _f64p]
        lib.smq_oracle_logits_contig.restype = ctypes.c_int
        lib.smq_oracle_logits_contig.argtypes = [
            ctypes.c_int, ctypes.c_int, _u8p, ctypes.c_float, _u16p, _u8p, _u8p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _f64p]
        lib.smq_oracle_candidate_mask.restype = ctypes.c_int
        lib.smq_oracle_candidate_mask.argtypes = [
            ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int64, _u8p]
        lib.smq_oracle_topk.restype = ctypes.c_int
        lib.smq_oracle_topk.argtypes = [ctypes.c_int64, _f64p, _u8p, ctypes.c_int, _i32p]
        lib.smq_oracle_expand.restype = ctypes.c_int
        lib.smq_oracle_expand.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int64, ctypes.c_int,
            _i32p, _i32p]
        lib.smq_oracle_encode_e2m1.restype = ctypes.c_uint8
        lib.smq_oracle_encode_e2m1.argtypes = [ctypes.c_double]
        lib.smq_oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.smq_oracle_encode_e4m3.argtypes = [ctypes.c_double]
        lib.smq_oracle_encode_bf16.restype = ctypes.c_uint16
        lib.smq_oracle_encode_bf16.argtypes = [ctypes.c_float]
        lib.smq_oracle_quantize_k_token.restype = ctypes.c_int
        lib.smq_oracle_quantize_k_token.argtypes = [ctypes.c_int, _u16p, _u8p, _u8p]
        lib.smq_oracle_write_k_cache.restype = ctypes.c_int
        lib.smq_oracle_write_k_cache.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, _i64p, ctypes.c_int64, _u8p,
                                                 ctypes.c_int64]
        lib.smq_oracle_quantize_q.restype = ctypes.c_int
        lib.smq_oracle_quantize_q.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, _f32p, _u8p, _f32p, _u16p]
        lib.smq_oracle_source_blocks.restype = ctypes.c_int
        lib.smq_oracle_source_blocks.argtypes = [ctypes.c_int64, _f64p, ctypes.c_int, ctypes.c_int, _f64p, _i32p]
        lib.smq_oracle_gather.restype = ctypes.c_int
        lib.smq_oracle_gather.argtypes = [
            ctypes.c_int, ctypes.c_int, _u8p, ctypes.c_int64, _i32p, ctypes.c_int64,
            ctypes.c_int64, _u8p, _u8p]
        self.lib = lib

    # -- element decoders ---------------------------------------------------
    def e4m3(self, code: int) -> float:
        return self.lib.smq_oracle_e4m3(code)

    def e2m1(self, nibble: int) -> float:
        return self.lib.smq_oracle_e2m1(nibble)

    def ue8m0(self, code: int) -> float:
        return self.lib.smq_oracle_ue8m0(code)

    def bf16(self, bits: int) -> float:
        return self.lib.smq_oracle_bf16(bits)

    # -- element encoders and producers ------------------------------------
    def encode_e2m1(self, v: float) -> int:
        return self.lib.smq_oracle_encode_e2m1(v)

    def encode_e4m3(self, v: float) -> int:
        return self.lib.smq_oracle_encode_e4m3(v)

    def encode_bf16(self, f: float) -> int:
        return self.lib.smq_oracle_encode_bf16(f)

    def quantize_k_token(self, k_bf16: np.ndarray):
        """One key [D] (bf16 bits) -> (packed E2M1 values [D/2], UE8M0 scales [D/32])."""
        k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
        d = k.shape[0]
        vals = np.empty(d // 2, dtype=np.uint8)
        scl = np.empty(d // 32, dtype=np.uint8)
        if self.lib.smq_oracle_quantize_k_token(d, _ptr(k, _u16p), _ptr(vals, _u8p), _ptr(scl, _u8p)) != 0:
            raise ValueError("oracle: non-finite key")
        return vals, scl

    def write_k_cache(self, k_bf16: np.ndarray, slot_mapping: np.ndarray, cache: np.ndarray, page_size: int):
        """Quantise keys [ntok, D] (bf16 bits) into the paged cache in place, token t to slot
        slot_mapping[t] (page * page_size + offset; negative: skipped)."""
        k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert cache.flags["C_CONTIGUOUS"] and cache.dtype == np.uint8
        rc = self.lib.smq_oracle_write_k_cache(k.shape[1], page_size, _ptr(k, _u16p), _ptr(slots, _i64p),
                                               k.shape[0], _ptr(cache, _u8p), cache.shape[0])
        if rc != 0:
            raise ValueError("oracle: slot past the cache or a non-finite key")

    def quantize_q(self, q_bf16: np.ndarray, w: np.ndarray):
        """Query rows [R, H, D] (bf16 bits) and weights [R, H] float32 -> (E4M3 codes [R, H, D],
        float32 scales [R], bf16 weights [R, H])."""
        q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
        w = np.ascontiguousarray(w, dtype=np.float32)
        R, H, D = q.shape
        q8 = np.empty((R, H, D), dtype=np.uint8)
        sc = np.empty(R, dtype=np.float32)
        wb = np.empty((R, H), dtype=np.uint16)
        for r in range(R):
            rc = self.lib.smq_oracle_quantize_q(H, D, _ptr(q[r], _u16p), _ptr(w[r], _f32p), _ptr(q8[r], _u8p),
                                                _ptr(sc[r:], _f32p), _ptr(wb[r], _u16p))
            if rc != 0:
                raise ValueError(f"oracle: non-finite query or weight in row {r}")
        return q8, sc, wb

    def source_blocks(self, logits: np.ndarray, cbs: int, ncb: int):
        """A row's dense logits [L] -> (its ncb published blocks, each block's maximum logit)."""
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        L = len(logits)
        nb = (L + cbs - 1) // cbs
        scores = np.empty(max(nb, 1), dtype=np.float64)
        cand = np.empty(ncb, dtype=np.int32)
        if self.lib.smq_oracle_source_blocks(L, _ptr(logits, _f64p), cbs, ncb, _ptr(scores, _f64p),
                                             _ptr(cand, _i32p)) != 0:
            raise MemoryError("oracle source blocks")
        return cand, scores[:nb]

    # -- per-row primitives -------------------------------------------------
    def logits_paged(self, inp, r: int, p0: int, p1: int) -> np.ndarray:
        """Dense logits of decode row r over sequence positions [p0, p1)."""
        g = inp.geom
        out = np.empty(max(0, p1 - p0), dtype=np.float64)
        q = np.ascontiguousarray(inp.q[r])
        w = np.ascontiguousarray(inp.weights[r])
        bt = np.ascontiguousarray(inp.block_table[inp.row_indices[r]])
        rc = self.lib.smq_oracle_logits_paged(
            g.num_heads, g.head_dim, g.page_size, _ptr(q, _u8p), float(inp.q_scale[r]),
            _ptr(w, _u16p), _ptr(inp.k_cache, _u8p), inp.k_cache.shape[0], _ptr(bt, _i32p),
            bt.shape[0], p0, p1, _ptr(out, _f64p))
        if rc != 0:
            raise ValueError(f"oracle: row {r} reads outside the cache or a non-finite value")
        return out

    def logits_contig(self, inp, k_values, k_scales, r: int, p0: int, p1: int) -> np.ndarray:
        """Dense logits of prefill row r over positions [p0, p1) relative to ks."""
        g = inp.geom
        out = np.empty(max(0, p1 - p0), dtype=np.float64)
        q = np.ascontiguousarray(inp.q[r])
        w = np.ascontiguousarray(inp.weights[r])
        rc = self.lib.smq_oracle_logits_contig(
            g.num_heads, g.head_dim, _ptr(q, _u8p), float(inp.q_scale[r]), _ptr(w, _u16p),
            _ptr(k_values, _u8p), _ptr(k_scales, _u8p), k_values.shape[0],
            int(inp.cu_seqlen_ks[r]), p0, p1, _ptr(out, _f64p))
        if rc != 0:
            raise ValueError(f"oracle: row {r} reads outside the workspace or a non-finite value")
        return out

    def candidate_mask(self, cbs: int, cand: np.ndarray, L: int) -> np.ndarray:
        cand = np.ascontiguousarray(cand, dtype=np.int32)
        valid = np.empty(max(L, 0), dtype=np.uint8)
        self.lib.smq_oracle_candidate_mask(cbs, len(cand), _ptr(cand, _i32p), L, _ptr(valid, _u8p))
        return valid

    def topk(self, logits: np.ndarray, valid: np.ndarray, k: int) -> np.ndarray:
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        valid = np.ascontiguousarray(valid, dtype=np.uint8)
        out = np.empty(k, dtype=np.int32)
        rc = self.lib.smq_oracle_topk(len(logits), _ptr(logits, _f64p), _ptr(valid, _u8p), k,
                                      _ptr(out, _i32p))
        if rc != 0:
            raise MemoryError("oracle top-k")
        return out

    def expand(self, cbs: int, sbkv: int, cand: np.ndarray, L: int, nsb: int):
        cand = np.ascontiguousarray(cand, dtype=np.int32)
        si = np.empty(nsb, dtype=np.int32)
        end = np.zeros(1, dtype=np.int32)
        rc = self.lib.smq_oracle_expand(cbs, sbkv, len(cand), _ptr(cand, _i32p), L, nsb,
                                        _ptr(si, _i32p), _ptr(end, _i32p))
        if rc != 0:
            raise ValueError("oracle expansion: bad sub-block size or too many sub-blocks")
        return si, int(end[0])

    def gather_seq(self, k_cache, page_size: int, head_dim: int, bt_row, seq_len: int):
        bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
        vals = np.empty((seq_len, head_dim // 2), dtype=np.uint8)
        scl = np.empty((seq_len, head_dim // 32), dtype=np.uint8)
        rc = self.lib.smq_oracle_gather(head_dim, page_size, _ptr(k_cache, _u8p), k_cache.shape[0],
                                        _ptr(bt_row, _i32p), len(bt_row), seq_len,
                                        _ptr(vals, _u8p), _ptr(scl, _u8p))
        if rc != 0:
            raise ValueError("oracle gather: page id out of range")
        return vals, scl


# --------------------------------------------------------------------------
# Row-level reference results
# --------------------------------------------------------------------------

_default = None
_default_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _default_lock:
        if _default is None:
            _default = Oracle()
        return _default


def sparse_block_kv(page_size: int, cbs: int) -> int:
    """The sub-block size both sides use: the largest of 128, 64, 32, 16 that
    divides the page size and the candidate block size.  This is our reading
    of ``pick_sparse_block_kv`` (sparse_indexer.py, builder ``__init__``): the
    pages require that the page size is a multiple of it and that it splits
    a candidate block, and they do not show the value it picks."""
    for s in (128, 64, 32, 16):
        if page_size % s == 0 and cbs % s == 0:
            return s
    raise ValueError("page_size and candidate_block_size need a common power-of-two divisor >= 16")


class RowResult:
    __slots__ = ("L", "logits", "valid", "topk", "sparse_indices", "end", "positions")

    def __init__(self, L, logits, valid, topk, sparse_indices, end, positions):
        self.L = L                      # row context length (ke - ks)
        self.logits = logits            # float64 logits (dense over [0, L), or at `positions`)
        self.valid = valid              # uint8 mask over [0, L) (dense mode) or None
        self.topk = topk                # int32 [k], -1 padded
        self.sparse_indices = sparse_indices  # int32 [nsb]
        self.end = end                  # valid column count
        self.positions = positions      # int64 positions of the columns, in column order


def _columns(si: np.ndarray, end: int, sbkv: int) -> np.ndarray:
    """Positions of the sparse columns in column order, truncated at end."""
    subs = si[si >= 0].astype(np.int64)
    pos = (subs[:, None] * sbkv + np.arange(sbkv)[None, :]).reshape(-1)
    return pos[:end]


def _row_reference(orc: Oracle, inp, r: int, mode: str, contig=None) -> RowResult:
    g = inp.geom
    sbkv = sparse_block_kv(g.page_size, g.candidate_block_size)
    nsb = g.candidate_topk_blocks * (g.candidate_block_size // sbkv)
    if contig is None:
        L = int(inp.row_ke[r])
    else:
        L = int(inp.cu_seqlen_ke[r]) - int(inp.cu_seqlen_ks[r])
    L = max(L, 0)
    si, end = orc.expand(g.candidate_block_size, sbkv, inp.candidate_blocks[r], L, nsb)
    pos = _columns(si, end, sbkv)

    def logits_range(p0, p1):
        if contig is None:
            return orc.logits_paged(inp, r, p0, p1)
        return orc.logits_contig(inp, contig[0], contig[1], r, p0, p1)

    if mode == "dense":
        logits = logits_range(0, L)
        valid = orc.candidate_mask(g.candidate_block_size, inp.candidate_blocks[r], L)
        top = orc.topk(logits, valid, g.topk)
        return RowResult(L, logits, valid, top, si, end, pos)
    if mode == "sparse":
        # candidate-only: score just the expanded columns, then the same top-k
        col_logits = np.empty(len(pos), dtype=np.float64)
        for i, s in enumerate(si[si >= 0]):
            p0 = int(s) * sbkv
            p1 = min(p0 + sbkv, L)
            a = i * sbkv
            col_logits[a:a + (p1 - p0)] = logits_range(p0, p1)
        full = np.zeros(L, dtype=np.float64)
        valid = np.zeros(L, dtype=np.uint8)
        full[pos] = col_logits
        valid[pos] = 1
        top = orc.topk(full, valid, g.topk)
        return RowResult(L, col_logits, None, top, si, end, pos)
    raise ValueError(mode)


def reference_rows(inp, rows: Optional[Iterable[int]] = None, mode: str = "sparse",
                   threads: Optional[int] = None, contig=None, orc: Optional[Oracle] = None):
    """Oracle results for the given rows of a DecodeInputs (contig=None) or a
    PrefillInputs (contig=(k_values, k_scales) from the oracle gather).

    mode="dense" scores every position of the row's context and masks
    (the definition); mode="sparse" scores only the candidate columns.
    """
    orc = orc or default()
    rows = list(range(inp.rows)) if rows is None else list(rows)
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(lambda r: _row_reference(orc, inp, r, mode, contig), rows))
    return dict(zip(rows, res))


def source_rows(inp, rows: Optional[Iterable[int]] = None, threads: Optional[int] = None,
                orc: Optional[Oracle] = None):
    """The candidate source of decode rows: dense logits over each row's whole
    context, then its published blocks. Returns {row: (cand [ncb], block
    scores, dense logits)}."""
    orc = orc or default()
    g = inp.geom
    rows = list(range(inp.rows)) if rows is None else list(rows)

    def one(r):
        L = max(int(inp.row_ke[r]), 0)
        logits = orc.logits_paged(inp, r, 0, L)
        cand, scores = orc.source_blocks(logits, g.candidate_block_size, g.candidate_topk_blocks)
        return cand, scores, logits

    with ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 1) as ex:
        res = list(ex.map(one, rows))
    return dict(zip(rows, res))


def gather_reference(inp, orc: Optional[Oracle] = None):
    """Oracle paged -> contiguous gather of every sequence of a PrefillInputs."""
    orc = orc or default()
    g = inp.geom
    total = inp.total_len
    vals = np.empty((total, g.head_dim // 2), dtype=np.uint8)
    scl = np.empty((total, g.head_dim // 32), dtype=np.uint8)
    for s in range(len(inp.cu_seq_lens) - 1):
        a, b = int(inp.cu_seq_lens[s]), int(inp.cu_seq_lens[s + 1])
        v, sc = orc.gather_seq(inp.k_cache, g.page_size, g.head_dim, inp.seq_block_table[s], b - a)
        vals[a:b] = v
        scl[a:b] = sc
    return vals, scl
