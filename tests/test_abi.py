"""The C-ABI library loads and exports every entry point include/*.h declares;
argument validation answers before any CUDA work (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

from selective_state_space_113_b300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    from selective_state_space_113_b300 import _native
    return _native.lib


def declared_symbols():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        names += re.findall(r"SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_symbols()
    for want in ("ssm_scan_fwd", "ssm_step", "ssm_device_status", "ssm_status_string",
                 "ssm_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_abi_version_and_status_strings(lib):
    assert lib.ssm_abi_version() == 1
    for code in range(-8, 1):
        s = lib.ssm_status_string(code)
        assert s and s != b"unknown status"
    assert lib.ssm_status_string(12345) == b"unknown status"


FAKE = 0x10000  # 64 KiB-aligned fake device address; validation never dereferences it


def scan(lib, u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, y=FAKE, h=None, batch=0, L=4,
         D=8, N=16, dtype=1, bias=None, Dskip=None, z=None):
    return lib.ssm_scan_fwd(u, delta, bias, A, B, C, Dskip, z, y, h, batch, L, D, N, dtype, None)


def step(lib, state=FAKE, u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, y=FAKE, batch=0, D=8,
         N=16, dtype=1):
    return lib.ssm_step(state, u, delta, None, A, B, C, None, None, y, batch, D, N, dtype, None)


def test_scan_argument_validation(lib):
    assert scan(lib) == 0                      # batch == 0: nothing to do
    for k in ("A",):
        assert scan(lib, **{k: None}) == -1    # A has D*N elements even when batch == 0
    for k in ("u", "delta", "B", "C", "y"):
        assert scan(lib, **{k: None}) == 0     # empty tensors may be NULL
        assert scan(lib, batch=1, **{k: None}) == -1
    assert scan(lib, batch=-1) == -2
    assert scan(lib, L=-1) == -2
    assert scan(lib, D=-1) == -2
    assert scan(lib, N=0) == -2
    assert scan(lib, N=257) == -5
    assert scan(lib, dtype=2) == -3
    assert scan(lib, batch=1 << 40, L=1 << 40) == -2   # overflow
    assert scan(lib, u=FAKE + 1) == -4                 # bf16 needs 2-byte alignment
    assert scan(lib, u=FAKE + 2) == 0                  # element-aligned is accepted
    assert scan(lib, u=FAKE + 2, dtype=0) == -4        # f32 needs 4-byte alignment
    assert scan(lib, A=FAKE + 2) == -4
    assert scan(lib, h=FAKE + 1) == -4


def test_step_argument_validation(lib):
    assert step(lib) == 0
    assert step(lib, A=None) == -1
    for k in ("state", "u", "delta", "B", "C", "y"):
        assert step(lib, **{k: None}) == 0
        assert step(lib, batch=1, **{k: None}) == -1
    assert step(lib, batch=-1) == -2
    assert step(lib, N=0) == -2
    assert step(lib, N=300) == -5
    assert step(lib, dtype=-1) == -3
    assert step(lib, state=FAKE + 2) == -4
