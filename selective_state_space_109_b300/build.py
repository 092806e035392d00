"""Builds libssmscan.so in-tree with nvcc for sm_103a (B300).

    python -m selective_state_space_109_b300.build [--force] [--verbose]

The CUDA runtime is linked statically, so the library loads on a machine
without a GPU (the C ABI's argument checks work there); the driver is only
needed once a call reaches the device.
"""
from __future__ import annotations

import argparse
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libssmscan.so")
SOURCES = [os.path.join(CSRC, f) for f in ("ssm_scan.cu", "scan_ws_bf16.cu", "scan_ws_f32.cu", "alu_probe.cu", "ssd.cu")]
OBJDIR = os.path.join(HERE, "_build")
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
    [os.path.join(INCLUDE, "ssm_scan.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Relocatable device code: the kernel translation units share the library's
# device error word; each compiles on its own (in parallel), then nvcc links
# the device code and the shared library.
COMPILE_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-rdc=true",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]
LINK_FLAGS = ARCH + ["-shared", "-rdc=true", "-cudart", "static"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in DEPS if os.path.exists(f))


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    from concurrent.futures import ThreadPoolExecutor
    os.makedirs(OBJDIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(OBJDIR, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc()] + COMPILE_FLAGS + (["-Xptxas=-v"] if ptxas_info else []) + \
            ["-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    cmd = [nvcc()] + LINK_FLAGS + ["-o", LIB + ".tmp"] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    sys.exit(main())
