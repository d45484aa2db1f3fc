"""Builds libpsr.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery)."""
from __future__ import annotations

import os
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libpsr.so")
LIB_TRACE = os.path.join(HERE, "libpsr_trace.so")  # same library with per-role cycle counters
LIB_PAIRS = os.path.join(HERE, "libpsr_pairs.so")  # same library with CTA-pair compute units for d = 128
# variant -> (extra nvcc defines, output)
VARIANTS = {"": ([], LIB), "trace": (["-DPSR_TRACE=1"], LIB_TRACE), "pairs": (["-DPSR_PAIRS=1"], LIB_PAIRS)}
SOURCES = [os.path.join(CSRC, f) for f in ("psr_ring_attn.cu", "psr_ring_attn_bwd.cu", "psr_ag_gemm.cu", "psr_gemm_rs.cu",
                                            "psr_noalloc.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f)
                  for f in ("psr_device.cuh", "psr_schedule.h", "psr_control.cuh", "psr_gemm_tile.cuh", "psr_internal.h")] + [
    os.path.join(ROOT, "include", "psr.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in DEPS)


def build(force: bool = False, verbose: bool = False, trace: bool = False, variant: str = "") -> str:
    """Compile the CUDA sources into persistent_sm_ring_gb300/libpsr.so, or a variant of it:
    "trace" (libpsr_trace.so, per-role cycle counters; also trace=True) or "pairs"
    (libpsr_pairs.so, CTA-pair compute units for d = 128)."""
    if trace:
        variant = "trace"
    defines, lib = VARIANTS[variant]
    with _lock:
        if not force and not needs_build(lib):
            return lib
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
               *defines, *SOURCES, "-o", tmp]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
        if verbose:
            print(res.stderr)
        os.replace(tmp, lib)
        return lib
