"""The C-ABI library without a GPU: it builds, loads, exports exactly what
include/smq.h declares, its structs match the binding, and the host-side
validation rejects bad arguments before any device work."""

import ctypes
import os
import re
import subprocess

import pytest

import sparse_attention_top_expand_gb300 as smq
from sparse_attention_top_expand_gb300.csrc import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smq.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return smq.load_library()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"SMQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for required in ("sparse_mqa_logits_topk_decode", "sparse_mqa_logits_topk_prefill_chunk",
                     "sparse_mqa_candidate_expand", "sparse_mqa_gather_k"):
        assert required in names
    assert sorted(smq.EXPORTED) == names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", smq.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out of the library
    assert {n for n in exported if not n.startswith("_")} == set(_declared())


def test_struct_layouts_match_binding(tmp_path):
    prog = tmp_path / "sizes.c"
    fields = {
        "smq_plan_desc": smq.SMQPlanDesc, "smq_plan_info": smq.SMQPlanInfo,
        "smq_decode_args": smq.SMQDecodeArgs, "smq_prefill_args": smq.SMQPrefillArgs,
        "smq_source_args": smq.SMQSourceArgs,
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "smq.h"', 'int main(void) {']
    for cname, cls in fields.items():
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname}.{fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for cname, cls in fields.items():
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert int(got[f"{cname}.{fname}"]) == getattr(cls, fname).offset, f"{cname}.{fname}"


def _desc(**kw):
    d = dict(num_heads=64, head_dim=128, page_size=64, candidate_block_size=128, candidate_topk_blocks=32,
             topk=2048, sparse_block_kv=0, max_rows=64, device=0)
    d.update(kw)
    return smq.SMQPlanDesc(ctypes.sizeof(smq.SMQPlanDesc), d["num_heads"], d["head_dim"], d["page_size"],
                           d["candidate_block_size"], d["candidate_topk_blocks"], d["topk"], d["sparse_block_kv"],
                           d["max_rows"], d["device"])


@pytest.mark.parametrize("bad,code", [
    (dict(num_heads=12), smq.SMQ_ERR_UNSUPPORTED),        # not a multiple of 8
    (dict(num_heads=256), smq.SMQ_ERR_UNSUPPORTED),
    (dict(head_dim=64), smq.SMQ_ERR_UNSUPPORTED),
    (dict(page_size=0), smq.SMQ_ERR_INVALID_ARG),
    (dict(candidate_block_size=0), smq.SMQ_ERR_INVALID_ARG),   # not a two-level indexer model
    (dict(candidate_topk_blocks=0), smq.SMQ_ERR_INVALID_ARG),
    (dict(topk=0), smq.SMQ_ERR_INVALID_ARG),
    (dict(topk=4097), smq.SMQ_ERR_INVALID_ARG),            # more than the sparse columns
    (dict(page_size=40, candidate_block_size=40), smq.SMQ_ERR_UNSUPPORTED),  # no power-of-two sub-block
    (dict(page_size=32, sparse_block_kv=64), smq.SMQ_ERR_INVALID_ARG),       # page not a multiple of it
    (dict(sparse_block_kv=24), smq.SMQ_ERR_UNSUPPORTED),
    (dict(candidate_topk_blocks=513), smq.SMQ_ERR_UNSUPPORTED),
    (dict(candidate_topk_blocks=256), smq.SMQ_ERR_UNSUPPORTED),  # 32768 sparse columns
    (dict(max_rows=0), smq.SMQ_ERR_INVALID_ARG),
    (dict(max_rows=20000), smq.SMQ_ERR_UNSUPPORTED),
    (dict(device=-1), smq.SMQ_ERR_INVALID_ARG),
])
def test_plan_create_rejects_bad_geometry(lib, bad, code):
    h = ctypes.c_void_p()
    d = _desc(**bad)
    assert lib.smq_plan_create(ctypes.byref(d), ctypes.byref(h)) == code
    assert not h.value


def test_plan_create_struct_size_checked(lib):
    d = _desc()
    d.struct_size = 8
    h = ctypes.c_void_p()
    assert lib.smq_plan_create(ctypes.byref(d), ctypes.byref(h)) == smq.SMQ_ERR_INVALID_ARG


def test_valid_geometry_reaches_the_device_check(lib):
    """A valid descriptor passes validation; without a usable sm_103 device
    the call reports CUDA / unsupported instead of creating a plan."""
    h = ctypes.c_void_p()
    rc = lib.smq_plan_create(ctypes.byref(_desc()), ctypes.byref(h))
    assert rc in (smq.SMQ_OK, smq.SMQ_ERR_CUDA, smq.SMQ_ERR_UNSUPPORTED)
    if rc == smq.SMQ_OK:
        lib.smq_plan_destroy(h)


def test_null_arguments_rejected(lib):
    assert lib.sparse_mqa_logits_topk_decode(None, None, None) == smq.SMQ_ERR_INVALID_ARG
    assert lib.sparse_mqa_logits_topk_prefill_chunk(None, None, None) == smq.SMQ_ERR_INVALID_ARG
    assert lib.sparse_mqa_candidate_expand(None, None, None, None, 1, None, None, None, 0, None) == \
        smq.SMQ_ERR_INVALID_ARG
    assert lib.sparse_mqa_gather_k(None, None, 1, None, 1, None, 1, 1, None, None, None, 0, None) == \
        smq.SMQ_ERR_INVALID_ARG
    code = ctypes.c_int32()
    assert lib.smq_get_status(None, None, ctypes.byref(code)) == smq.SMQ_ERR_INVALID_ARG


def test_error_strings(lib):
    for c in (0, 1, 2, 3, 4, 8, 16, 24):
        assert lib.smq_error_string(c)
    assert b"range" in lib.smq_error_string(smq.SMQ_ERR_BOUNDS)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    mod = importlib.reload(smq)
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError):
        mod.load_library(str(tmp_path / "missing.so"))
    importlib.reload(smq)
