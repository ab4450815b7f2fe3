"""Build the CDB shared library in-tree for sm_103a (GB300).

``python -m continuous_depth_batching_gb300.build`` compiles every source in
``csrc/`` with nvcc in parallel and links ``_build/libcdb.so``.  Objects are
rebuilt only when a source or header is newer.  The CUDA runtime is linked
statically so the library loads on machines without a GPU (the CPU tests
check its exports); the driver API is reached through the runtime's entry
point query, never linked.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libcdb.so")

SOURCES = [
    "sched.cpp",
    "sim.cpp",
    "planner.cpp",
    "engine.cu",
    "kernels.cu",
    "attention.cu",
    "attention_prefill_tc.cu",
    "gemm_simt.cu",
    "gemm_tc.cu",
    "attention_noalloc.cu",
    "tmap.cu",
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found; the CDB library needs the CUDA toolkit to build")


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    inc = os.path.join(ROOT, "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _compile(src: str, verbose: bool) -> str:
    nvcc = _nvcc()
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, "obj", src + ".o")
    newest = max([os.path.getmtime(path)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest:
        return obj
    os.makedirs(os.path.dirname(obj), exist_ok=True)
    cmd = [nvcc, "-c", path, "-o", obj, "-O3", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")] + ARCH
    if src.endswith(".cu"):
        cmd += ["--expt-relaxed-constexpr"]
        if verbose:
            cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False) -> str:
    """Compile (if stale) and link the library; returns the .so path."""
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max(1, min(len(SOURCES), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs):
        return LIB
    cmd = [_nvcc(), "-shared", "-o", LIB + ".tmp"] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
