"""Builds the in-tree CUDA libraries for sm_103a with nvcc.

libmoe.so        the engine (csrc/moe_abi.cu and the kernels it includes)
libmoe_synth.so  the device twin of the synthetic-input generator

Both are compiled in parallel, one -gencode (compute_103a / sm_103a), -O3,
-lineinfo, no fast-math; a library is rebuilt when a source or header is
newer than it.
"""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

LIBMOE = os.path.join(PKG, "libmoe.so")
LIBSYNTH = os.path.join(PKG, "libmoe_synth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static"]


def _nvcc() -> str:
    for p in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if p and os.path.exists(p):
            return p
    return "nvcc"


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def targets():
    hdrs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return [
        (LIBMOE, os.path.join(CSRC, "moe_abi.cu"), hdrs),
        (LIBSYNTH, os.path.join(CSRC, "moe_synth.cu"), [os.path.join(INCLUDE, "moe_synth.h")]),
    ]


def build(force: bool = False, extra_flags=()) -> list:
    """Compile every stale library; returns the list of library paths."""
    procs = []
    for out, src, hdrs in targets():
        if force or _stale(out, [src] + hdrs):
            tmp = out + f".tmp{os.getpid()}"
            cmd = [_nvcc()] + ARCH + FLAGS + list(extra_flags) + ["-o", tmp, src]
            procs.append((out, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                          stderr=subprocess.STDOUT, text=True)))
    errors = []
    for out, tmp, cmd, p in procs:
        log, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{' '.join(cmd)}\n{log}")
        else:
            os.replace(tmp, out)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    return [t[0] for t in targets()]


if __name__ == "__main__":
    print(build(force=True))
