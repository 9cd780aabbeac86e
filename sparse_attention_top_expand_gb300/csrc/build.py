"""Build libsmq.so, the sm_103a C-ABI library, in-tree with nvcc.

Three translation units are compiled in parallel and then linked. Only the
SMQ_API entry points of include/smq.h are exported.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libsmq.so")
TRACE_LIB = os.path.join(PKG, "libsmq_trace.so")  # -DSMQ_TRACE: phase timestamps (include/smq_trace.h)
SOURCES = ["smq_api.cu", "smq_kernels.cu", "smq_producers.cu", "smq_prefill.cu"]
HEADERS = ["smq_kernels.cuh", "smq_ptx.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE, "-I", HERE,
]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(HERE, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, h)
                                                                for h in ("smq.h", "smq_trace.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), trace: bool = False) -> str:
    """Compile libsmq.so, or with trace=True the tracing build libsmq_trace.so."""
    out = TRACE_LIB if trace else LIB
    if not force and not _stale(out):
        return out
    if trace:
        extra_flags = (*extra_flags, "-DSMQ_TRACE")
    objdir = os.path.join(PKG, "_build", "trace" if trace else "lib")
    os.makedirs(objdir, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [_nvcc(), *NVCC_FLAGS, *extra_flags, "-c", os.path.join(HERE, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    for cmd, p in procs:
        log, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(log)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    tmp = out + ".tmp"
    link = [_nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp]
    subprocess.run(link, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
