"""Builds libgqa_b300.so in-tree with nvcc for sm_103a.

    python -m grouped_query_attention_11_b300.build [--verbose-ptxas]

The library is two translation units (csrc/gqa_api.cu: the C ABI with the
warp-level kernels; csrc/gqa_umma.cu: the tensor-core kernel), compiled in
parallel and linked against the static CUDA runtime, so it loads on a machine
without a GPU driver; the driver is only needed when a compute call runs.
"""
from __future__ import annotations

import argparse
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgqa_b300.so")
SOURCES = [os.path.join(CSRC, "gqa_api.cu"), os.path.join(CSRC, "gqa_umma.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cuh", ".h"))] + [
    os.path.join(INCLUDE, "gqa.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand)
                     or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compiles each translation unit (in parallel) and links the library."""
    if not force and up_to_date():
        return LIB
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(CSRC, os.path.basename(src) + tag + ".o")
        cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-c",
               "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, "-o", obj,
               src]
        if ptxas_verbose:
            cmd[1:1] = ["-Xptxas", "-v"]
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd)))
    try:
        for cmd, proc in procs:
            if proc.wait() != 0:
                raise subprocess.CalledProcessError(proc.returncode, cmd)
        tmp = LIB + tag
        subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o",
                        tmp, *objs], check=True)
        os.replace(tmp, LIB)
    finally:
        # a failed compile leaves the others running: stop them before the
        # objects they would still write are cleaned up
        for _, proc in procs:
            if proc.poll() is None:
                proc.kill()
            proc.wait()
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force or a.verbose_ptxas,
                ptxas_verbose=a.verbose_ptxas))
    return 0


if __name__ == "__main__":
    sys.exit(main())
