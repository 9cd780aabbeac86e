"""Comparison rules between the CUDA path and the oracle (test infrastructure).

Logits: a column passes when |gpu - ref| <= max(ATOL, RTOL * |ref|).  The
oracle is exact to ~1e-15 relative (double arithmetic over products that
are exact in double); the GPU accumulates the same products in fp32, so any
deviation above ~1e-5 relative means a bug, far inside the bound.

bf16 logits (the optional bf16 output): each is the fp32 logit rounded to
the nearest-even bfloat16, so a column passes when |gpu - ref| <=
max(ATOL, RTOL * |ref|) + 2^-8 * |ref|: with 8 significant bits, half a
bf16 step is at most 2^-8 of the value.

Top-k: the output order inside a row is not specified by the pages, so rows
are compared as sets.  The count of ids must be min(k, |valid|) and the rest
-1; ids must be distinct valid positions; an id that one side picked and the
other did not must lie within the logit tolerance of the oracle's k-th value
(several answers are correct when values tie there).
"""

from __future__ import annotations

import numpy as np

ATOL = 1e-2
RTOL = 1e-3


def tol(ref):
    return np.maximum(ATOL, RTOL * np.abs(ref))


def check_logits(gpu: np.ndarray, ref: np.ndarray, what: str = "logits") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if gpu.shape != ref.shape:
        raise AssertionError(f"{what}: shape {gpu.shape} != {ref.shape}")
    if not np.all(np.isfinite(gpu)):
        bad = np.flatnonzero(~np.isfinite(gpu))[:5]
        raise AssertionError(f"{what}: non-finite at columns {bad.tolist()}")
    err = np.abs(gpu - ref)
    bad = err > tol(ref)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {len(ref)} columns out of tolerance; first at {i}: "
            f"gpu={gpu[i]!r} ref={ref[i]!r}")


def check_logits_bf16(gpu: np.ndarray, ref: np.ndarray, what: str = "bf16 logits") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if gpu.shape != ref.shape:
        raise AssertionError(f"{what}: shape {gpu.shape} != {ref.shape}")
    bound = tol(ref) + np.abs(ref) * 2.0 ** -8
    bad = ~(np.abs(gpu - ref) <= bound)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {len(ref)} columns out of tolerance; first at {i}: "
                             f"gpu={gpu[i]!r} ref={ref[i]!r}")


def check_topk(gpu_ids: np.ndarray, row, k: int, what: str = "topk") -> None:
    """Compare one row's GPU ids with an oracle RowResult."""
    gpu_ids = np.asarray(gpu_ids, dtype=np.int64)
    ref_ids = np.asarray(row.topk, dtype=np.int64)
    n_valid = int(row.end)
    want = min(k, n_valid)
    sel = gpu_ids[:want]
    if len(gpu_ids) != k:
        raise AssertionError(f"{what}: {len(gpu_ids)} ids, expected {k}")
    if np.any(gpu_ids[want:] != -1):
        raise AssertionError(f"{what}: expected -1 after {want} ids, got {gpu_ids[want:want + 8].tolist()}")
    if np.any(sel < 0):
        raise AssertionError(f"{what}: {int((sel < 0).sum())} of the first {want} ids are -1")
    if len(np.unique(sel)) != want:
        raise AssertionError(f"{what}: repeated ids")
    valid_pos = np.asarray(row.positions, dtype=np.int64)
    if not np.all(np.isin(sel, valid_pos)):
        bad = sel[~np.isin(sel, valid_pos)][:5]
        raise AssertionError(f"{what}: ids outside the candidate columns: {bad.tolist()}")
    ref_sel = ref_ids[:want]
    if want < n_valid:
        # ref logit of each candidate position
        lut = dict(zip(valid_pos.tolist(), _row_logits_at(row, valid_pos)))
        v_k = lut[int(ref_sel[-1])]
        diff = np.setxor1d(sel, ref_sel)
        for p in diff.tolist():
            if abs(lut[p] - v_k) > max(ATOL, RTOL * abs(v_k)):
                raise AssertionError(
                    f"{what}: position {p} (ref logit {lut[p]!r}) differs from the oracle's set "
                    f"and is not tied with the k-th value {v_k!r}")
    else:
        if set(sel.tolist()) != set(ref_sel.tolist()):
            raise AssertionError(f"{what}: all valid positions must be selected")


def _row_logits_at(row, positions):
    if row.valid is not None:  # dense mode: logits over [0, L)
        return np.asarray(row.logits)[positions]
    return np.asarray(row.logits)  # sparse mode: logits in column order == positions order
