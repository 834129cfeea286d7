"""Builds libkvring.so in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared
library with the CUDA runtime linked statically (the library needs only the
driver at run time).  No CMake, no torch extension machinery.

Usage: python -m ring_kv_cache_gb300.build  (or ``build()`` from Python)
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libkvring.so")
BUILD = os.path.join(HERE, "_build")
SOURCES = ["kvring_host.cu", "kvring_cache.cu", "kvring_attn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, nvcc: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    return obj, p.stderr


def build(verbose: bool = False) -> str:
    """Compile every translation unit and link libkvring.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, nvcc), SOURCES))
    logs = []
    for (obj, log), src in zip(results, SOURCES):
        logs.append(f"== {src}\n{log}")
    cmd = [nvcc, *ARCH, "-shared", "-o", OUT + ".tmp", *[o for o, _ in results], "-cudart", "static"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(OUT + ".tmp", OUT)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if verbose:
        print("\n".join(logs))
    return OUT


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(OUT)
