"""Build libssmscan.so in-tree with nvcc for sm_103a.

``python -m selective_state_space_113_b300.build`` compiles the single
translation unit ``csrc/api.cu`` (which includes every kernel file) into
``selective_state_space_113_b300/libssmscan.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libssmscan.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise FileNotFoundError("nvcc not found")


def sources() -> list[str]:
    out = [os.path.join(ROOT, "include", "ssmscan.h")]
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")):
            out.append(os.path.join(CSRC, f))
    return out


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(out: str = LIB, extra=(), verbose: bool = False, force: bool = False) -> str:
    """Compile the library; returns its path.  ``extra`` adds nvcc flags."""
    if not force and not extra and up_to_date(out):
        return out
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-Xptxas", "-warn-spills", *extra,
           "-o", out, os.path.join(CSRC, "api.cu")]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv,
          extra=tuple(a for a in sys.argv[1:] if a != "--force"))
