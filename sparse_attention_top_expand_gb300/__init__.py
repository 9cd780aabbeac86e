"""Python binding of libsmq, the GB300 (sm_103a) candidate-block sparse
MQA-logits top-k indexer.

The functions carry the names of the C entry points in include/smq.h. They
only marshal arguments: they check devices, dtypes and contiguity, pass
data pointers and the current CUDA stream, and turn error codes into
exceptions. Every step of the computation runs in the library's kernels.
PyTorch provides device memory and streams only. If the library is
missing, the import of any entry point raises; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmq.so")

SMQ_OK = 0
SMQ_ERR_INVALID_ARG = 1
SMQ_ERR_UNSUPPORTED = 2
SMQ_ERR_WORKSPACE_TOO_SMALL = 3
SMQ_ERR_CUDA = 4
SMQ_ERR_BOUNDS = 8
SMQ_ERR_TIMEOUT = 16
SMQ_NOALLOC_SCRATCH_BYTES = 8 << 20  # logits scratch of sparse_mqa_logits_topk_decode_noalloc

_c_i32 = ctypes.c_int32
_c_u32 = ctypes.c_uint32
_c_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class SMQPlanDesc(ctypes.Structure):
    _fields_ = [("struct_size", _c_u32), ("num_heads", _c_i32), ("head_dim", _c_i32), ("page_size", _c_i32),
                ("candidate_block_size", _c_i32), ("candidate_topk_blocks", _c_i32), ("topk", _c_i32),
                ("sparse_block_kv", _c_i32), ("max_rows", _c_i32), ("device", _c_i32)]


class SMQPlanInfo(ctypes.Structure):
    _fields_ = [("struct_size", _c_u32), ("sparse_block_kv", _c_i32), ("num_sparse_blocks", _c_i32),
                ("num_sparse_cols", _c_i32), ("page_bytes", _c_i32), ("num_sms", _c_i32)]


class SMQDecodeArgs(ctypes.Structure):
    _fields_ = [("struct_size", _c_u32), ("rows", _c_i32), ("q", _vp), ("q_scale", _vp), ("weights", _vp),
                ("k_cache", _vp), ("num_pages", _c_i64), ("block_table", _vp), ("bt_rows", _c_i32),
                ("bt_stride", _c_i32), ("row_indices", _vp), ("row_ke", _vp), ("candidate_blocks", _vp),
                ("topk_out", _vp), ("topk_ld", _c_i32), ("sparse_indices", _vp), ("end", _vp),
                ("expansion_ready", _c_i32), ("col_indices", _vp), ("logits_out", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("profile_events", _vp * 4), ("logits_out_bf16", _vp)]


class SMQPrefillArgs(ctypes.Structure):
    _fields_ = [("struct_size", _c_u32), ("rows", _c_i32), ("q", _vp), ("q_scale", _vp), ("weights", _vp),
                ("k_values", _vp), ("k_scales", _vp), ("total_len", _c_i64), ("cu_seqlen_ks", _vp),
                ("cu_seqlen_ke", _vp), ("candidate_blocks", _vp), ("topk_out", _vp), ("topk_ld", _c_i32),
                ("sparse_indices", _vp), ("end", _vp), ("expansion_ready", _c_i32), ("col_indices", _vp),
                ("logits_out", _vp), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
                ("profile_events", _vp * 4), ("logits_out_bf16", _vp)]


class SMQSourceArgs(ctypes.Structure):
    _fields_ = [("struct_size", _c_u32), ("rows", _c_i32), ("q", _vp), ("q_scale", _vp), ("weights", _vp),
                ("k_cache", _vp), ("num_pages", _c_i64), ("block_table", _vp), ("bt_rows", _c_i32),
                ("bt_stride", _c_i32), ("row_indices", _vp), ("row_ke", _vp), ("max_context", _c_i32),
                ("candidate_blocks", _vp), ("block_scores", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t)]


EXPORTED = [
    "smq_plan_create", "smq_plan_destroy", "smq_plan_get_info", "smq_workspace_size", "smq_workspace_init",
    "smq_prefill_workspace_size",
    "smq_get_status", "smq_error_string", "sparse_mqa_candidate_expand", "sparse_mqa_logits_topk_decode",
    "sparse_mqa_logits_topk_prefill_chunk", "sparse_mqa_gather_k", "sparse_mqa_logits_topk_decode_noalloc",
    "sparse_mqa_write_k_cache", "sparse_mqa_quantize_q", "smq_source_workspace_size",
    "sparse_mqa_candidate_source_decode", "smq_plan_set_wait_limit", "smq_plan_inject_stall",
]

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsmq.so (built by __graft_entry__.build() or csrc/build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsmq.so is not built ({path}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.smq_plan_create.argtypes = [P(SMQPlanDesc), P(_vp)]
    lib.smq_plan_destroy.argtypes = [_vp]
    lib.smq_plan_get_info.argtypes = [_vp, P(SMQPlanInfo)]
    lib.smq_workspace_size.argtypes = [_vp, _c_i32, P(ctypes.c_size_t)]
    lib.smq_prefill_workspace_size.argtypes = [_vp, _c_i32, ctypes.c_int64, P(ctypes.c_size_t)]
    lib.smq_workspace_init.argtypes = [_vp, _vp, ctypes.c_size_t, _vp]
    lib.smq_get_status.argtypes = [_vp, _vp, P(_c_i32)]
    lib.smq_error_string.argtypes = [ctypes.c_int]
    lib.smq_error_string.restype = ctypes.c_char_p
    lib.sparse_mqa_candidate_expand.argtypes = [_vp, _vp, _vp, _vp, _c_i32, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.sparse_mqa_logits_topk_decode.argtypes = [_vp, P(SMQDecodeArgs), _vp]
    lib.sparse_mqa_logits_topk_decode_noalloc.argtypes = [_vp, P(SMQDecodeArgs), _vp]
    lib.sparse_mqa_logits_topk_prefill_chunk.argtypes = [_vp, P(SMQPrefillArgs), _vp]
    lib.sparse_mqa_gather_k.argtypes = [_vp, _vp, _c_i64, _vp, _c_i32, _vp, _c_i32, _c_i64, _vp, _vp, _vp,
                                        ctypes.c_size_t, _vp]
    lib.sparse_mqa_write_k_cache.argtypes = [_vp, _vp, _vp, _c_i64, _vp, _c_i64, _vp, ctypes.c_size_t, _vp]
    lib.sparse_mqa_quantize_q.argtypes = [_vp, _vp, _vp, _c_i32, _vp, _vp, _vp, _vp]
    lib.smq_source_workspace_size.argtypes = [_vp, _c_i32, _c_i32, P(ctypes.c_size_t)]
    lib.smq_plan_set_wait_limit.argtypes = [_vp, _c_i64]
    lib.smq_plan_inject_stall.argtypes = [_vp, _c_i32]
    lib.sparse_mqa_candidate_source_decode.argtypes = [_vp, P(SMQSourceArgs), _vp]
    for name in EXPORTED:
        if name != "smq_error_string":
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


class SMQError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load_library().smq_error_string(code).decode()
        super().__init__(f"{where}: {msg} (code {code})")
        self.code = code


def _check(code: int, where: str) -> None:
    if code != SMQ_OK:
        raise SMQError(code, where)


def _ptr(t: Optional[torch.Tensor], dtypes, name: str, device=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _set_events(args, events) -> None:
    """Optional torch.cuda.Event / raw cudaEvent_t handles for the profile_events slots."""
    if events is None:
        return
    for i, ev in enumerate(events):
        if ev is None:
            continue
        args.profile_events[i] = ev.cuda_event if hasattr(ev, "cuda_event") else int(ev)


_U8 = (torch.uint8,)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_BF16 = (torch.bfloat16, torch.int16)


class Plan:
    """A validated geometry (smq_plan_create); close() or GC frees it."""

    def __init__(self, num_heads: int, page_size: int, candidate_block_size: int, candidate_topk_blocks: int,
                 topk: int, max_rows: int, head_dim: int = 128, sparse_block_kv: int = 0,
                 device: Optional[int] = None):
        lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        self.device_index = int(device)
        self.device = torch.device("cuda", self.device_index)
        d = SMQPlanDesc(ctypes.sizeof(SMQPlanDesc), num_heads, head_dim, page_size, candidate_block_size,
                        candidate_topk_blocks, topk, sparse_block_kv, max_rows, self.device_index)
        h = _vp()
        _check(lib.smq_plan_create(ctypes.byref(d), ctypes.byref(h)), "smq_plan_create")
        self.handle = h
        info = SMQPlanInfo()
        info.struct_size = ctypes.sizeof(SMQPlanInfo)
        _check(lib.smq_plan_get_info(h, ctypes.byref(info)), "smq_plan_get_info")
        self.num_heads = num_heads
        self.head_dim = head_dim
        self.page_size = page_size
        self.candidate_block_size = candidate_block_size
        self.candidate_topk_blocks = candidate_topk_blocks
        self.topk = topk
        self.max_rows = max_rows
        self.sparse_block_kv = info.sparse_block_kv
        self.num_sparse_blocks = info.num_sparse_blocks
        self.num_sparse_cols = info.num_sparse_cols
        self.page_bytes = info.page_bytes
        self.num_sms = info.num_sms

    def set_wait_limit(self, ns: int) -> None:
        """Every pipeline wait of later calls gives up after ns nanoseconds (default 2 s)."""
        _check(load_library().smq_plan_set_wait_limit(self.handle, int(ns)), "smq_plan_set_wait_limit")

    def inject_stall(self, tile: int) -> None:
        """Failure-path tests: withhold tile `tile`'s hand-off in the first CTA (-1: none)."""
        _check(load_library().smq_plan_inject_stall(self.handle, int(tile)), "smq_plan_inject_stall")

    def workspace_size(self, rows: int) -> int:
        n = ctypes.c_size_t()
        _check(load_library().smq_workspace_size(self.handle, rows, ctypes.byref(n)), "smq_workspace_size")
        return n.value

    def prefill_workspace_size(self, rows: int, total_len: int) -> int:
        n = ctypes.c_size_t()
        _check(load_library().smq_prefill_workspace_size(self.handle, rows, total_len, ctypes.byref(n)),
               "smq_prefill_workspace_size")
        return n.value

    def workspace(self, rows: Optional[int] = None, stream=None, total_len: Optional[int] = None) -> torch.Tensor:
        """Allocate (here, by torch) and zero a workspace for calls of up to `rows` rows; with `total_len`, one
        that also holds the window-major prefill scratch for chunks of up to that many workspace rows."""
        rows = self.max_rows if rows is None else rows
        n = self.workspace_size(rows) if total_len is None else self.prefill_workspace_size(rows, total_len)
        ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        smq_workspace_init(self, ws, stream)
        return ws

    def close(self) -> None:
        if getattr(self, "handle", None):
            load_library().smq_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def smq_workspace_init(plan: Plan, workspace: torch.Tensor, stream=None) -> None:
    _check(load_library().smq_workspace_init(plan.handle, _ptr(workspace, _U8, "workspace"), workspace.numel(),
                                             _stream(stream)), "smq_workspace_init")


def smq_get_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream, return the device status bits and clear them."""
    code = _c_i32()
    _check(load_library().smq_get_status(_ptr(workspace, _U8, "workspace"), _stream(stream), ctypes.byref(code)),
           "smq_get_status")
    return code.value


def sparse_mqa_candidate_expand(plan: Plan, candidate_blocks, row_ks, row_ke, sparse_indices, end, workspace,
                                stream=None) -> None:
    rows = int(row_ke.shape[0])
    dev = plan.device
    _check(load_library().sparse_mqa_candidate_expand(
        plan.handle, _ptr(candidate_blocks, _I32, "candidate_blocks", dev), _ptr(row_ks, _I32, "row_ks", dev),
        _ptr(row_ke, _I32, "row_ke", dev), rows, _ptr(sparse_indices, _I32, "sparse_indices", dev),
        _ptr(end, _I32, "end", dev), _ptr(workspace, _U8, "workspace", dev), workspace.numel(), _stream(stream)),
        "sparse_mqa_candidate_expand")


def _decode_args(plan: Plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke, candidate_blocks,
                 topk_out, sparse_indices, end, workspace, expansion_ready, col_indices, logits_out,
                 logits_out_bf16=None):
    dev = plan.device
    a = SMQDecodeArgs()
    a.struct_size = ctypes.sizeof(SMQDecodeArgs)
    a.rows = int(q.shape[0])
    a.q = _ptr(q, _U8, "q", dev)
    a.q_scale = _ptr(q_scale, _F32, "q_scale", dev)
    a.weights = _ptr(weights, _BF16, "weights", dev)
    a.k_cache = _ptr(k_cache, _U8, "k_cache", dev)
    a.num_pages = int(k_cache.shape[0])
    a.block_table = _ptr(block_table, _I32, "block_table", dev)
    a.bt_rows = int(block_table.shape[0])
    a.bt_stride = int(block_table.shape[1])
    a.row_indices = _ptr(row_indices, _I32, "row_indices", dev)
    a.row_ke = _ptr(row_ke, _I32, "row_ke", dev)
    a.candidate_blocks = _ptr(candidate_blocks, _I32, "candidate_blocks", dev)
    a.topk_out = _ptr(topk_out, _I32, "topk_out", dev)
    a.topk_ld = int(topk_out.shape[1])
    a.sparse_indices = _ptr(sparse_indices, _I32, "sparse_indices", dev)
    a.end = _ptr(end, _I32, "end", dev)
    a.expansion_ready = 1 if expansion_ready else 0
    a.col_indices = _ptr(col_indices, _I32, "col_indices", dev)
    a.logits_out = _ptr(logits_out, _F32, "logits_out", dev)
    a.logits_out_bf16 = _ptr(logits_out_bf16, _BF16, "logits_out_bf16", dev)
    if workspace is not None:
        a.workspace = _ptr(workspace, _U8, "workspace", dev)
        a.workspace_bytes = workspace.numel()
    return a


def sparse_mqa_logits_topk_decode(plan: Plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke,
                                  candidate_blocks, topk_out, sparse_indices, end, workspace,
                                  expansion_ready: bool = False, col_indices=None, logits_out=None,
                                  stream=None, profile_events=None, logits_out_bf16=None) -> None:
    a = _decode_args(plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke, candidate_blocks,
                     topk_out, sparse_indices, end, workspace, expansion_ready, col_indices, logits_out,
                     logits_out_bf16)
    _set_events(a, profile_events)
    _check(load_library().sparse_mqa_logits_topk_decode(plan.handle, ctypes.byref(a), _stream(stream)),
           "sparse_mqa_logits_topk_decode")


class DecodeCall:
    """sparse_mqa_logits_topk_decode with its arguments marshalled once, for a
    loop that calls it again and again on the same buffers (their contents may
    change between calls, their addresses and shapes may not). Each call goes
    through the same C entry point."""

    def __init__(self, plan: Plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke, candidate_blocks,
                 topk_out, sparse_indices, end, workspace, expansion_ready: bool = False, col_indices=None,
                 logits_out=None):
        self.plan = plan
        self.args = _decode_args(plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke,
                                 candidate_blocks, topk_out, sparse_indices, end, workspace, expansion_ready,
                                 col_indices, logits_out)
        # the buffers stay alive as long as the call
        self._keep = (q, q_scale, weights, k_cache, block_table, row_indices, row_ke, candidate_blocks, topk_out,
                      sparse_indices, end, workspace, col_indices, logits_out)
        self._fn = load_library().sparse_mqa_logits_topk_decode
        self._ref = ctypes.byref(self.args)

    def __call__(self, stream=None) -> None:
        rc = self._fn(self.plan.handle, self._ref, _stream(stream))
        if rc != 0:
            _check(rc, "sparse_mqa_logits_topk_decode")


def sparse_mqa_logits_topk_decode_noalloc(plan: Plan, q, q_scale, weights, k_cache, block_table, row_indices,
                                          row_ke, candidate_blocks, topk_out, sparse_indices, end,
                                          expansion_ready: bool = False, col_indices=None, logits_out=None,
                                          stream=None, logits_out_bf16=None) -> None:
    """Paged decode on the library's static scratch: no workspace argument,
    at most 8 MiB of fp32 logits (rows x sparse columns), calls must not
    overlap on the GPU, device-detected errors are not reported."""
    a = _decode_args(plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke, candidate_blocks,
                     topk_out, sparse_indices, end, None, expansion_ready, col_indices, logits_out, logits_out_bf16)
    _check(load_library().sparse_mqa_logits_topk_decode_noalloc(plan.handle, ctypes.byref(a), _stream(stream)),
           "sparse_mqa_logits_topk_decode_noalloc")


def sparse_mqa_logits_topk_prefill_chunk(plan: Plan, q, q_scale, weights, k_values, k_scales, cu_seqlen_ks,
                                         cu_seqlen_ke, candidate_blocks, topk_out, sparse_indices, end, workspace,
                                         expansion_ready: bool = False, col_indices=None, logits_out=None,
                                         stream=None, profile_events=None, logits_out_bf16=None) -> None:
    dev = plan.device
    a = SMQPrefillArgs()
    a.struct_size = ctypes.sizeof(SMQPrefillArgs)
    a.rows = int(q.shape[0])
    a.q = _ptr(q, _U8, "q", dev)
    a.q_scale = _ptr(q_scale, _F32, "q_scale", dev)
    a.weights = _ptr(weights, _BF16, "weights", dev)
    a.k_values = _ptr(k_values, _U8, "k_values", dev)
    a.k_scales = _ptr(k_scales, _U8, "k_scales", dev)
    a.total_len = int(k_values.shape[0])
    a.cu_seqlen_ks = _ptr(cu_seqlen_ks, _I32, "cu_seqlen_ks", dev)
    a.cu_seqlen_ke = _ptr(cu_seqlen_ke, _I32, "cu_seqlen_ke", dev)
    a.candidate_blocks = _ptr(candidate_blocks, _I32, "candidate_blocks", dev)
    a.topk_out = _ptr(topk_out, _I32, "topk_out", dev)
    a.topk_ld = int(topk_out.shape[1])
    a.sparse_indices = _ptr(sparse_indices, _I32, "sparse_indices", dev)
    a.end = _ptr(end, _I32, "end", dev)
    a.expansion_ready = 1 if expansion_ready else 0
    a.col_indices = _ptr(col_indices, _I32, "col_indices", dev)
    a.logits_out = _ptr(logits_out, _F32, "logits_out", dev)
    a.logits_out_bf16 = _ptr(logits_out_bf16, _BF16, "logits_out_bf16", dev)
    a.workspace = _ptr(workspace, _U8, "workspace", dev)
    a.workspace_bytes = workspace.numel()
    _set_events(a, profile_events)
    _check(load_library().sparse_mqa_logits_topk_prefill_chunk(plan.handle, ctypes.byref(a), _stream(stream)),
           "sparse_mqa_logits_topk_prefill_chunk")


def sparse_mqa_gather_k(plan: Plan, k_cache, block_table, cu_seq_lens, total_len: int, k_values, k_scales,
                        workspace, stream=None) -> None:
    dev = plan.device
    _check(load_library().sparse_mqa_gather_k(
        plan.handle, _ptr(k_cache, _U8, "k_cache", dev), int(k_cache.shape[0]),
        _ptr(block_table, _I32, "block_table", dev), int(block_table.shape[1]),
        _ptr(cu_seq_lens, _I32, "cu_seq_lens", dev), int(cu_seq_lens.shape[0]) - 1, int(total_len),
        _ptr(k_values, _U8, "k_values", dev), _ptr(k_scales, _U8, "k_scales", dev),
        _ptr(workspace, _U8, "workspace", dev), workspace.numel(), _stream(stream)), "sparse_mqa_gather_k")


def sparse_mqa_write_k_cache(plan: Plan, k, slot_mapping, k_cache, workspace, stream=None) -> None:
    """Quantise keys [ntok, D] (bf16) into the paged MXFP4 cache at slot_mapping [ntok] (int64)."""
    dev = plan.device
    _check(load_library().sparse_mqa_write_k_cache(
        plan.handle, _ptr(k, _BF16, "k", dev), _ptr(slot_mapping, (torch.int64,), "slot_mapping", dev),
        int(k.shape[0]), _ptr(k_cache, _U8, "k_cache", dev), int(k_cache.shape[0]),
        _ptr(workspace, _U8, "workspace", dev), workspace.numel(), _stream(stream)), "sparse_mqa_write_k_cache")


def sparse_mqa_quantize_q(plan: Plan, q, weights, q_fp8, q_scale, weights_bf16, stream=None) -> None:
    """Quantise query rows [R, H, D] (bf16) to E4M3 with a float scale per row, and float
    weights [R, H] to bf16."""
    dev = plan.device
    _check(load_library().sparse_mqa_quantize_q(
        plan.handle, _ptr(q, _BF16, "q", dev), _ptr(weights, _F32, "weights", dev), int(q.shape[0]),
        _ptr(q_fp8, _U8, "q_fp8", dev), _ptr(q_scale, _F32, "q_scale", dev),
        _ptr(weights_bf16, _BF16, "weights_bf16", dev), _stream(stream)), "sparse_mqa_quantize_q")


def smq_source_workspace_size(plan: Plan, rows: int, max_context: int) -> int:
    n = ctypes.c_size_t()
    _check(load_library().smq_source_workspace_size(plan.handle, rows, max_context, ctypes.byref(n)),
           "smq_source_workspace_size")
    return n.value


def sparse_mqa_candidate_source_decode(plan: Plan, q, q_scale, weights, k_cache, block_table, row_indices, row_ke,
                                       max_context: int, candidate_blocks, workspace, block_scores=None,
                                       stream=None) -> None:
    """The candidate source: dense scores over each row's context, then the row's
    candidate_topk_blocks best blocks of candidate_block_size positions."""
    dev = plan.device
    a = SMQSourceArgs()
    a.struct_size = ctypes.sizeof(SMQSourceArgs)
    a.rows = int(q.shape[0])
    a.q = _ptr(q, _U8, "q", dev)
    a.q_scale = _ptr(q_scale, _F32, "q_scale", dev)
    a.weights = _ptr(weights, _BF16, "weights", dev)
    a.k_cache = _ptr(k_cache, _U8, "k_cache", dev)
    a.num_pages = int(k_cache.shape[0])
    a.block_table = _ptr(block_table, _I32, "block_table", dev)
    a.bt_rows = int(block_table.shape[0])
    a.bt_stride = int(block_table.shape[1])
    a.row_indices = _ptr(row_indices, _I32, "row_indices", dev)
    a.row_ke = _ptr(row_ke, _I32, "row_ke", dev)
    a.max_context = int(max_context)
    a.candidate_blocks = _ptr(candidate_blocks, _I32, "candidate_blocks", dev)
    a.block_scores = _ptr(block_scores, _F32, "block_scores", dev)
    a.workspace = _ptr(workspace, _U8, "workspace", dev)
    a.workspace_bytes = workspace.numel()
    _check(load_library().sparse_mqa_candidate_source_decode(plan.handle, ctypes.byref(a), _stream(stream)),
           "sparse_mqa_candidate_source_decode")
