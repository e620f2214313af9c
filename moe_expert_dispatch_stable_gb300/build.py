"""Build the MoE-LoRA CUDA library for sm_103a (in-tree, no cmake).

Each translation unit is compiled in parallel with nvcc, then linked into
``libmoe_lora_gb300.so`` next to this file.  The C runtime is linked
statically; driver entry points (TMA descriptor encoding) are fetched at run
time through the runtime, so the library links no libcuda.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_lora_gb300.so")
# the debug build: every index read from a caller's routing buffer is checked before use
# (MOE_DEBUG=1; out-of-range indices set MOE_DEV_BAD_INDEX and are skipped)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmoe_lora_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["route.cu", "router.cu", "rowops.cu", "quant.cu", "packed.cu", "gemm_tc.cu", "gemm_wgrad.cu", "api.cu"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and shutil.which(cand) is None:
        raise RuntimeError("nvcc not found; the MoE-LoRA library needs the CUDA 13 toolkit")
    return cand


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "moe_lora.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile (if stale) and link the library (the debug build with debug=True);
    returns its path."""
    nvcc = _nvcc()
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    if debug:
        extra_flags = (*extra_flags, "-DMOE_DEBUG=1")
    os.makedirs(bdir, exist_ok=True)
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if _stale(o, s):
            jobs.append([nvcc, *_flags(extra_flags), "-c", s, "-o", o])
    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for msg in ex.map(run, jobs):
            if verbose and msg:
                print(msg, file=sys.stderr)
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
