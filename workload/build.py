"""Build the workload generator libraries in-tree.

libclkgen_host.so : gcc, host generator (also handed to the CPU oracle).
libclkgen_dev.so  : nvcc for sm_103a, device generator used by GPU tests and the benchmark.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def build_host(verbose: bool = False) -> str:
    out = os.path.join(HERE, "libclkgen_host.so")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-o", out, os.path.join(HERE, "gen_host.c")]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return out


def dev_cmd() -> list:
    out = os.path.join(HERE, "libclkgen_dev.so")
    return ["nvcc", ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
            "-o", out, os.path.join(HERE, "gen_device.cu")]


def build_dev(verbose: bool = False) -> str:
    cmd = dev_cmd()
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return cmd[cmd.index("-o") + 1]


if __name__ == "__main__":
    build_host(True)
    build_dev(True)
