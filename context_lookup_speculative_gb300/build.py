"""In-tree build of libclk.so (nvcc, sm_103a only; each .cu compiled in parallel)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libclk.so")
SOURCES = ["clk_api.cu", "clk_lookup.cu", "clk_verify.cu", "clk_sample.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
NVFLAGS = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           f"-I{INCLUDE}", f"-I{CSRC}"]


def _compile(src: str, extra, verbose: bool, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = ["nvcc", *NVFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    return obj


def build(verbose: bool = False, extra=(), out: str = LIB, build_dir: str = BUILD) -> str:
    """Compile every source for sm_103a and link libclk.so (next to this file
    unless `out` names another path)."""
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra), verbose, build_dir), SOURCES))
    cmd = ["nvcc", ARCH, "-shared", "-o", out, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(verbose=True, extra=["-Xptxas", "-v"] if os.environ.get("CLK_PTXAS_V") else [])
