"""libssmscan: the selective state-space scan (Mamba's S6 core) and its decode
step as hand-written CUDA kernels for B300 (sm_103a), behind a C ABI
(``include/ssmscan.h``).  This package holds the kernels (``csrc/``), their
in-tree build (``build.py``), the ctypes binding (``_native.py``, loaded on
first use) and the seeded workload generators (``workloads.py``).

The binding is imported lazily so that the workload generators stay usable on
machines without the built library; calling any entry point without the
library raises ImportError (there is no CPU fallback).
"""
from __future__ import annotations

__all__ = ["ssm_scan_fwd", "ssm_scan_fwd_disc", "ssm_conv_scan_fwd", "ssm_scan_bwd", "ssm_scan_fwd_ckpt", "ssm_scan_bwd_ckpt", "ssm_ssd_fwd", "ssm_scan_fwd_noalloc", "ssm_step", "ssm_device_status", "ssm_status_string",
           "ssm_abi_version", "ssm_unit_ceilings", "SsmError", "scan", "step"]


def __getattr__(name):
    if name in ("ssm_scan_fwd", "ssm_scan_fwd_disc", "ssm_conv_scan_fwd", "ssm_scan_bwd", "ssm_scan_fwd_ckpt", "ssm_scan_bwd_ckpt", "ssm_ssd_fwd", "SSM_DISC_ZOH", "SSM_DISC_EULER",
                "SSM_DISC_TRAPEZOID", "ssm_scan_fwd_noalloc", "ssm_step", "ssm_device_status", "ssm_status_string",
                "ssm_abi_version", "ssm_unit_ceilings", "SsmError", "lib", "LIB_PATH"):
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)


def scan(u, delta, dt_bias, A, B, C, Dskip=None, z=None, want_h_last=True, stream=None):
    """Allocate y (and h_last) and run ssm_scan_fwd; returns (y, h_last or None)."""
    import torch
    from ._native import ssm_scan_fwd
    y = torch.empty_like(u)
    h = (torch.empty((u.shape[0], u.shape[2], A.shape[-1]), device=u.device,
                     dtype=torch.float32) if want_h_last else None)
    ssm_scan_fwd(u, delta, dt_bias, A, B, C, Dskip, z, y, h, stream=stream)
    return y, h


def step(state, u, delta, dt_bias, A, B, C, Dskip=None, z=None, stream=None):
    """Allocate y and run ssm_step (state updated in place); returns y."""
    import torch
    from ._native import ssm_step
    y = torch.empty_like(u)
    ssm_step(state, u, delta, dt_bias, A, B, C, Dskip, z, y, stream=stream)
    return y
