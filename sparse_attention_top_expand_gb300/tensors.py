"""Move synthetic inputs (numpy, from synth.py) to device tensors and run the
library's entry points on them. This module only marshals data: it copies
arrays, allocates outputs and calls the binding.
"""

from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (Plan, sparse_mqa_candidate_expand, sparse_mqa_gather_k, sparse_mqa_logits_topk_decode,
               sparse_mqa_logits_topk_prefill_chunk)


def _t(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def plan_for(geom, max_rows: int, device=None) -> Plan:
    return Plan(num_heads=geom.num_heads, page_size=geom.page_size, candidate_block_size=geom.candidate_block_size,
                candidate_topk_blocks=geom.candidate_topk_blocks, topk=geom.topk, max_rows=max_rows,
                head_dim=geom.head_dim, device=device)


class DecodeDevice:
    """Device copies of a DecodeInputs plus output buffers."""

    def __init__(self, inp, plan: Plan, with_logits: bool = True, with_cols: bool = True,
                 with_logits_bf16: bool = False):
        dev = plan.device
        R = inp.rows
        self.rows = R
        self.q = _t(inp.q, dev)
        self.q_scale = _t(inp.q_scale, dev)
        self.weights = _t(inp.weights, dev)
        self.k_cache = _t(inp.k_cache, dev)
        self.block_table = _t(inp.block_table, dev)
        self.row_indices = _t(inp.row_indices, dev)
        self.row_ke = _t(inp.row_ke, dev)
        self.candidate_blocks = _t(inp.candidate_blocks, dev)
        self.topk_out = torch.full((R, plan.topk), -7, dtype=torch.int32, device=dev)
        self.sparse_indices = torch.full((R, plan.num_sparse_blocks), -7, dtype=torch.int32, device=dev)
        self.end = torch.full((R,), -7, dtype=torch.int32, device=dev)
        self.col_indices = torch.full((R, plan.topk), -7, dtype=torch.int32, device=dev) if with_cols else None
        self.logits = torch.full((R, plan.num_sparse_cols), float("nan"), dtype=torch.float32,
                                 device=dev) if with_logits else None
        self.logits_bf16 = torch.full((R, plan.num_sparse_cols), 0x7FC1, dtype=torch.int16,
                                      device=dev) if with_logits_bf16 else None
        self.workspace = plan.workspace(max(R, 1))

    def run(self, plan: Plan, expansion_ready: bool = False, stream=None) -> None:
        sparse_mqa_logits_topk_decode(plan, self.q, self.q_scale, self.weights, self.k_cache, self.block_table,
                                      self.row_indices, self.row_ke, self.candidate_blocks, self.topk_out,
                                      self.sparse_indices, self.end, self.workspace,
                                      expansion_ready=expansion_ready, col_indices=self.col_indices,
                                      logits_out=self.logits, stream=stream, logits_out_bf16=self.logits_bf16)

    def expand(self, plan: Plan, stream=None) -> None:
        sparse_mqa_candidate_expand(plan, self.candidate_blocks, None, self.row_ke, self.sparse_indices, self.end,
                                    self.workspace, stream=stream)


class PrefillDevice:
    """Device copies of a PrefillInputs (paged cache + gathered workspace) plus outputs. With window_major the
    workspace also holds the window-major path's scratch (the call then takes that path)."""

    def __init__(self, inp, plan: Plan, with_logits: bool = True, with_cols: bool = True,
                 with_logits_bf16: bool = False, window_major: bool = True):
        dev = plan.device
        R = inp.rows
        self.rows = R
        self.q = _t(inp.q, dev)
        self.q_scale = _t(inp.q_scale, dev)
        self.weights = _t(inp.weights, dev)
        self.k_cache = _t(inp.k_cache, dev)
        self.seq_block_table = _t(inp.seq_block_table, dev)
        self.cu_seq_lens = _t(inp.cu_seq_lens, dev)
        self.total_len = inp.total_len
        self.k_values = torch.zeros((self.total_len, inp.geom.head_dim // 2), dtype=torch.uint8, device=dev)
        self.k_scales = torch.zeros((self.total_len, inp.geom.head_dim // 32), dtype=torch.uint8, device=dev)
        self.ks = _t(inp.cu_seqlen_ks, dev)
        self.ke = _t(inp.cu_seqlen_ke, dev)
        self.candidate_blocks = _t(inp.candidate_blocks, dev)
        self.topk_out = torch.full((R, plan.topk), -7, dtype=torch.int32, device=dev)
        self.sparse_indices = torch.full((R, plan.num_sparse_blocks), -7, dtype=torch.int32, device=dev)
        self.end = torch.full((R,), -7, dtype=torch.int32, device=dev)
        self.col_indices = torch.full((R, plan.topk), -7, dtype=torch.int32, device=dev) if with_cols else None
        self.logits = torch.full((R, plan.num_sparse_cols), float("nan"), dtype=torch.float32,
                                 device=dev) if with_logits else None
        self.logits_bf16 = torch.full((R, plan.num_sparse_cols), 0x7FC1, dtype=torch.int16,
                                      device=dev) if with_logits_bf16 else None
        # sized for the window-major prefill path, or for the row-major one only
        self.workspace = plan.workspace(max(R, 1), total_len=self.total_len if window_major else None)

    def gather(self, plan: Plan, stream=None) -> None:
        sparse_mqa_gather_k(plan, self.k_cache, self.seq_block_table, self.cu_seq_lens, self.total_len,
                            self.k_values, self.k_scales, self.workspace, stream=stream)

    def run(self, plan: Plan, expansion_ready: bool = False, stream=None) -> None:
        sparse_mqa_logits_topk_prefill_chunk(plan, self.q, self.q_scale, self.weights, self.k_values, self.k_scales,
                                             self.ks, self.ke, self.candidate_blocks, self.topk_out,
                                             self.sparse_indices, self.end, self.workspace,
                                             expansion_ready=expansion_ready, col_indices=self.col_indices,
                                             logits_out=self.logits, stream=stream,
                                             logits_out_bf16=self.logits_bf16)


def to_numpy(t: Optional[torch.Tensor]):
    return None if t is None else t.detach().cpu().numpy()
