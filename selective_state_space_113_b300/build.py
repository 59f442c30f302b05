"""Build libssmscan.so in-tree with nvcc for sm_103a.

``python -m selective_state_space_113_b300.build`` compiles the single
translation unit ``csrc/api.cu`` (which includes every kernel file) into
``selective_state_space_113_b300/libssmscan.so``.  A build is skipped when the
library is current: when a stamp written by the last successful build (a
SHA-256 of the nvcc flags and of every source's contents, kept in ``_build/``)
matches, or, with no stamp, when no source is newer than the library.  So a
checkout that only rewrites files, changing their times but not their
contents, does not trigger the (several-minute) compile.
"""
from __future__ import annotations

import hashlib
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


# The nvcc flags after the compiler's path (no output or source path).  No
# --split-compile: the split optimiser gave slower code (the scan 4% slower,
# the SSD kernels 2-13%, with different register counts) for no shorter build on an
# 8-core host (about 6.5 minutes either way).
FLAGS = (*ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-warn-spills")


def command(out: str = LIB, extra=()) -> list[str]:
    return [nvcc_path(), *FLAGS, *extra, "-o", out, os.path.join(CSRC, "api.cu")]


def digest(cmd: list[str]) -> str:
    """SHA-256 of the compile flags (not the compiler's location) and of every
    source file's relative path and contents."""
    h = hashlib.sha256()
    h.update("\0".join(cmd[1:]).encode())
    for src in sources():
        h.update(b"\0" + os.path.relpath(src, ROOT).encode() + b"\0")
        with open(src, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def stamp_path(out: str = LIB) -> str:
    return os.path.join(ROOT, "_build", os.path.basename(out) + ".stamp")


def up_to_date(out: str = LIB, extra=()) -> bool:
    if not os.path.exists(out):
        return False
    stamp = stamp_path(out)
    if os.path.exists(stamp):
        with open(stamp) as fh:
            return fh.read().strip() == digest(command(out, extra))
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(out: str = LIB, extra=(), verbose: bool = False, force: bool = False) -> str:
    """Compile the library; returns its path.  ``extra`` adds nvcc flags."""
    if not force and not extra and up_to_date(out):
        return out
    cmd = command(out, extra)
    # the sources as compiled: hashed before nvcc reads them, so an edit
    # made while it runs leaves the stamp stale rather than wrong
    d = digest(cmd)
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    stamp = stamp_path(out)
    os.makedirs(os.path.dirname(stamp), exist_ok=True)
    with open(stamp, "w") as fh:
        fh.write(d + "\n")
    return out


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv,
          extra=tuple(a for a in sys.argv[1:] if a != "--force"))
