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
    for code in range(-9, 1):
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


def disc(lib, code, batch=0, **kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, y=FAKE)
    a.update(kw)
    return lib.ssm_scan_fwd_disc(a["u"], a["delta"], None, a["A"], a["B"], a["C"], None, None,
                                 a["y"], None, batch, 4, 8, 16, 1, code, None)


def test_disc_argument_validation(lib):
    for code in (0, 1, 2):
        assert disc(lib, code) == 0
    assert disc(lib, 3) == -5
    assert disc(lib, -1) == -5
    assert disc(lib, 1, batch=1, u=None) == -1
    assert disc(lib, 2, u=FAKE + 1) == -4


def conv(lib, w=FAKE, b=None, act=1, batch=0, x=FAKE, D=8):
    return lib.ssm_conv_scan_fwd(x, w, b, act, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE,
                                 None, batch, 4, D, 16, 1, None)


def test_conv_argument_validation(lib):
    assert conv(lib) == 0
    assert conv(lib, act=0) == 0
    assert conv(lib, w=None) == -1            # the filter is required when D > 0
    assert conv(lib, w=None, D=0) == 0
    assert conv(lib, act=2) == -5
    assert conv(lib, w=FAKE + 2) == -4        # float32 filter needs 4-byte alignment
    assert conv(lib, b=FAKE + 1) == -4
    assert conv(lib, batch=1, x=None) == -1


BWD_ARGS = ("u", "delta", "dt_bias", "A", "B", "C", "Dskip", "z", "dy", "dh_last", "du", "ddelta",
            "ddt_bias", "dA", "dB", "dC", "dDskip", "dz")


def bwd(lib, batch=1, L=4, D=8, N=16, dtype=1, **kw):
    a = {k: FAKE for k in BWD_ARGS}
    for k in ("dt_bias", "Dskip", "z", "dh_last", "ddt_bias", "dB", "dC", "dDskip", "dz"):
        a[k] = None
    a.update(kw)
    return lib.ssm_scan_bwd(*[a[k] for k in BWD_ARGS], batch, L, D, N, dtype, None)


def test_bwd_argument_validation(lib):
    """Only the rejections: a valid call clears the derivative sums with CUDA."""
    for k in ("u", "delta", "dy", "du", "ddelta", "B", "C", "A", "dA"):
        assert bwd(lib, **{k: None}) == -1, k
    assert bwd(lib, z=FAKE) == -1                       # z given without dz
    assert bwd(lib, batch=-1) == -2
    assert bwd(lib, N=0) == -2
    assert bwd(lib, N=257) == -5
    assert bwd(lib, dtype=2) == -3
    assert bwd(lib, batch=1 << 30, L=1 << 30, D=1) == -2   # index range of the workspace
    assert bwd(lib, dy=FAKE + 1) == -4
    assert bwd(lib, dz=FAKE + 1, z=FAKE) == -4
    assert bwd(lib, dB=FAKE + 2) == -4
    assert bwd(lib, dh_last=FAKE + 2) == -4


def ckpt_fwd(lib, batch=1, L=64, D=8, N=16, dtype=1, **kw):
    a = dict(u=FAKE, delta=FAKE, dt_bias=None, A=FAKE, B=FAKE, C=FAKE, Dskip=None, z=None, y=FAKE,
             h_last=None, ckpt=FAKE)
    a.update(kw)
    return lib.ssm_scan_fwd_ckpt(a["u"], a["delta"], a["dt_bias"], a["A"], a["B"], a["C"],
                                 a["Dskip"], a["z"], a["y"], a["h_last"], a["ckpt"], batch, L, D, N,
                                 dtype, None)


def ckpt_bwd(lib, batch=1, L=64, D=8, N=16, dtype=1, **kw):
    a = dict(u=FAKE, delta=FAKE, dt_bias=None, A=FAKE, B=FAKE, C=FAKE, Dskip=None, z=None, dy=FAKE,
             dh_last=None, ckpt=FAKE, du=FAKE, ddelta=FAKE, ddt_bias=None, dA=FAKE, dB=None,
             dC=None, dDskip=None, dz=None)
    a.update(kw)
    return lib.ssm_scan_bwd_ckpt(a["u"], a["delta"], a["dt_bias"], a["A"], a["B"], a["C"],
                                 a["Dskip"], a["z"], a["dy"], a["dh_last"], a["ckpt"], a["du"],
                                 a["ddelta"], a["ddt_bias"], a["dA"], a["dB"], a["dC"],
                                 a["dDskip"], a["dz"], batch, L, D, N, dtype, None)


def test_checkpoint_argument_validation(lib):
    """The checkpoint pair's rejections, all before anything is enqueued:
    checkpoints needed (L > 32) but NULL, misaligned, or a shape that the
    N == 16 kernels do not take; no channels is a no-op."""
    for fn in (ckpt_fwd, ckpt_bwd):
        assert fn(lib, ckpt=None) == -1, fn.__name__
        assert fn(lib, ckpt=FAKE + 4) == -4, fn.__name__
        assert fn(lib, N=7) == -5, fn.__name__
        assert fn(lib, D=4) == -5, fn.__name__              # a bf16 row of 8 bytes
        assert fn(lib, u=None) == -1, fn.__name__
    assert ckpt_fwd(lib, batch=0) == 0


def ssd(lib, batch=0, L=4, H=2, P=64, N=64, dtype=1, **kw):
    a = dict(x=FAKE, dt=FAKE, dt_bias=None, A=FAKE, B=FAKE, C=FAKE, Dskip=None, y=FAKE,
             h_last=None)
    a.update(kw)
    return lib.ssm_ssd_fwd(a["x"], a["dt"], a["dt_bias"], a["A"], a["B"], a["C"], a["Dskip"],
                           a["y"], a["h_last"], batch, L, H, P, N, dtype, None)


def test_ssd_argument_validation(lib):
    assert ssd(lib) == 0                     # no channels: nothing to do
    assert ssd(lib, A=None) == -1            # A has H elements even when batch == 0
    for k in ("x", "dt", "B", "C", "y"):
        assert ssd(lib, **{k: None}) == 0
        assert ssd(lib, batch=1, **{k: None}) == -1, k
    assert ssd(lib, P=0) == -2
    assert ssd(lib, H=-1) == -2
    assert ssd(lib, N=0) == -2
    assert ssd(lib, N=257) == -5
    assert ssd(lib, dtype=7) == -3
    assert ssd(lib, batch=1 << 40, L=1 << 40) == -2
    assert ssd(lib, x=FAKE + 1) == -4
    assert ssd(lib, dt_bias=FAKE + 2) == -4


def noalloc(lib, batch=0, L=4, D=8, h=None, **kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, y=FAKE)
    a.update(kw)
    return lib.ssm_scan_fwd_noalloc(a["u"], a["delta"], None, a["A"], a["B"], a["C"], None, None,
                                    a["y"], h, batch, L, D, 16, 1, None)


def test_noalloc_argument_validation(lib):
    assert noalloc(lib) == 0
    assert noalloc(lib, A=None) == -1
    assert noalloc(lib, batch=1, y=None) == -1
    assert noalloc(lib, batch=-1) == -2
    assert noalloc(lib, u=FAKE + 1) == -4
    # a fast-path problem whose carried states (64 bytes per channel without
    # h_last) cannot fit the fixed scratch is refused before any CUDA call
    assert noalloc(lib, batch=1024, D=8192) == -9


def test_ceilings_argument_validation(lib):
    buf = (ctypes.c_double * 3)()
    assert lib.ssm_unit_ceilings(None, 1, None) == -1
    assert lib.ssm_unit_ceilings(buf, 0, None) == -2
