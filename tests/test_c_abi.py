"""The boundary from plain C: a C99 program compiled against include/ssmscan.h
(with -Wall -Wextra -Werror -pedantic) links the library and gets the
documented answers from the calls that answer on the host (CPU only)."""
import os
import shutil
import subprocess

import pytest

from selective_state_space_113_b300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_caller(tmp_path):
    lib = libbuild.build()
    exe = str(tmp_path / "c_abi_check")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
                    lib, "-Wl,-rpath," + os.path.dirname(lib), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi check: ok" in r.stdout
