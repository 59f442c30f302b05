"""Calls in a new CUDA context: a C program (tests/c_ctx_reset.c) runs the
scan, the allocation-free scan, the decode step, the SSD form and the
backward, destroys its context with cudaDeviceReset, and runs them again.
What the library caches per device that belongs to a context (kernel
shared-memory limits, the workspace pool, the fixed scratch array's address)
must be set up again there, and every output must come out byte for byte the
same.  The program is also compiled on the CPU machine, where it cannot run."""
import os
import shutil
import subprocess

import pytest

from selective_state_space_113_b300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_program(tmp_path):
    lib = libbuild.build()
    exe = str(tmp_path / "c_ctx_reset")
    # C11: the CUDA runtime's own headers use anonymous unions
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    os.path.join(ROOT, "tests", "c_ctx_reset.c"), lib,
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(CUDA, "lib64"),
                    "-o", exe], check=True)
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_ctx_reset_program_builds(tmp_path):
    assert os.path.exists(build_program(tmp_path))


@pytest.mark.gpu
@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_calls_after_device_reset(tmp_path):
    exe = build_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ctx reset check: ok" in r.stdout
