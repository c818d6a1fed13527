"""Build ``libnf4bwd.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel to ``_build/*.o``; the objects are
linked with the static CUDA runtime into ``backward_gemm_gb300/libnf4bwd.so``.
The driver API (tensor-map encoding) is reached through the runtime's
driver-entry-point query, so nothing links against libcuda.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnf4bwd.so")

SOURCES = ["nf4_quant.cu", "nf4_gemm.cu", "rms_norm_bwd.cu"]
HEADERS = ["ptx.cuh", "nf4_dequant.cuh", "nf4_common.h", "pair_kernel.cuh", "prepass.cuh",
           "host_plan.cuh", "small_m_host.cuh", "nf4_small_m.cuh", "nf4_trace.cuh",
           "dense_gemm.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "--expt-relaxed-constexpr", "-diag-suppress", "1160"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(INCLUDE, "nf4bwd.h"), os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _defines() -> list[str]:
    """Diagnostic builds: NF4BWD_DEFINES="NF4_TRACE" (clock probes, read back
    through nf4_debug_set_trace) or "NF4_PROGRESS" (per-role progress counters,
    nf4_debug_set_progress), comma-separated.  Product builds define neither."""
    names = [d.strip() for d in os.environ.get("NF4BWD_DEFINES", "").split(",") if d.strip()]
    allowed = {"NF4_TRACE", "NF4_PROGRESS"}
    bad = [d for d in names if d not in allowed]
    if bad:
        raise RuntimeError(f"NF4BWD_DEFINES: unknown {bad}; allowed {sorted(allowed)}")
    return [f"-D{d}" for d in names]


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *_defines(), *extra, "-c", os.path.join(CSRC, src), "-o",
           obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if "-Xptxas" in extra:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library if it is missing or older than its sources."""
    if not force and not is_stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
