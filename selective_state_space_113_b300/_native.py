"""ctypes binding of libssmscan (include/ssmscan.h), argument marshalling only.

Each function has the C entry point's name and argument order.  Tensor
arguments are torch CUDA tensors (or None for an optional NULL); sizes and the
dtype code are taken from the tensors' shapes and dtypes; ``stream`` defaults
to torch's current CUDA stream.  A non-zero status raises ``SsmError``.  There
is no fallback: if the shared library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssmscan.so")

SSM_F32, SSM_BF16 = 0, 1
STATUS = {0: "SSM_OK", -1: "SSM_ERR_NULL", -2: "SSM_ERR_SIZE", -3: "SSM_ERR_DTYPE",
          -4: "SSM_ERR_ALIGN", -5: "SSM_ERR_UNSUPPORTED", -6: "SSM_ERR_CUDA",
          -7: "SSM_ERR_NOMEM", -8: "SSM_ERR_TIMEOUT", -9: "SSM_ERR_SCRATCH"}
EXPORTS = ("ssm_scan_fwd", "ssm_scan_fwd_disc", "ssm_conv_scan_fwd", "ssm_scan_bwd",
           "ssm_scan_fwd_ckpt", "ssm_scan_bwd_ckpt",
           "ssm_ssd_fwd", "ssm_scan_fwd_noalloc", "ssm_step",
           "ssm_device_status", "ssm_status_string", "ssm_abi_version", "ssm_unit_ceilings")
SSM_DISC_ZOH, SSM_DISC_EULER, SSM_DISC_TRAPEZOID = 0, 1, 2


class SsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_text(status)})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssmscan.so is not built ({LIB_PATH}); run "
                          "`python -m selective_state_space_113_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.ssm_scan_fwd.restype = ci
    lib.ssm_scan_fwd.argtypes = [vp] * 10 + [i64] * 4 + [ci, vp]
    lib.ssm_scan_fwd_disc.restype = ci
    lib.ssm_scan_fwd_disc.argtypes = [vp] * 10 + [i64] * 4 + [ci, ci, vp]
    lib.ssm_conv_scan_fwd.restype = ci
    lib.ssm_conv_scan_fwd.argtypes = [vp] * 3 + [ci] + [vp] * 9 + [i64] * 4 + [ci, vp]
    lib.ssm_scan_bwd.restype = ci
    lib.ssm_scan_bwd.argtypes = [vp] * 18 + [i64] * 4 + [ci, vp]
    lib.ssm_scan_fwd_ckpt.restype = ci
    lib.ssm_scan_fwd_ckpt.argtypes = [vp] * 11 + [i64] * 4 + [ci, vp]
    lib.ssm_scan_bwd_ckpt.restype = ci
    lib.ssm_scan_bwd_ckpt.argtypes = [vp] * 19 + [i64] * 4 + [ci, vp]
    lib.ssm_ssd_fwd.restype = ci
    lib.ssm_ssd_fwd.argtypes = [vp] * 9 + [i64] * 5 + [ci, vp]
    lib.ssm_scan_fwd_noalloc.restype = ci
    lib.ssm_scan_fwd_noalloc.argtypes = [vp] * 10 + [i64] * 4 + [ci, vp]
    lib.ssm_step.restype = ci
    lib.ssm_step.argtypes = [vp] * 10 + [i64] * 3 + [ci, vp]
    lib.ssm_device_status.restype = ci
    lib.ssm_device_status.argtypes = [vp]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [ci]
    lib.ssm_abi_version.restype = ci
    lib.ssm_unit_ceilings.restype = ci
    lib.ssm_unit_ceilings.argtypes = [ctypes.POINTER(ctypes.c_double), ci, vp]
    if lib.ssm_abi_version() != 1:
        raise ImportError("libssmscan ABI version mismatch")
    return lib


lib = _load()


def status_text(status: int) -> str:
    return lib.ssm_status_string(int(status)).decode()


def ssm_status_string(status: int) -> str:
    return status_text(status)


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SsmError(status, where)


def ssm_scan_fwd(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, stream=None) -> None:
    """y, h_last <- selective scan of (u, delta, dt_bias, A, B, C, Dskip, z)."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_fwd(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip),
                            _p(z), _p(y), _p(h_last), batch, L, D, N, _dtype_code(u),
                            _stream(stream)), "ssm_scan_fwd")


def ssm_scan_fwd_disc(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, disc, stream=None) -> None:
    """ssm_scan_fwd with the discretisation `disc` (SSM_DISC_ZOH, _EULER or
    _TRAPEZOID) of the input term."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_fwd_disc(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip),
                                 _p(z), _p(y), _p(h_last), batch, L, D, N, _dtype_code(u),
                                 int(disc), _stream(stream)), "ssm_scan_fwd_disc")


def ssm_conv_scan_fwd(x, conv_w, conv_b, act, delta, dt_bias, A, B, C, Dskip, z, y, h_last,
                      stream=None) -> None:
    """y, h_last <- ssm_scan_fwd of u = act(causal width-4 depthwise conv of x
    with conv_w [D, 4] and conv_b [D]); act 1 is SiLU, 0 none."""
    batch, L, D = x.shape
    N = A.shape[-1]
    _check(lib.ssm_conv_scan_fwd(_p(x), _p(conv_w), _p(conv_b), int(act), _p(delta),
                                 _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip), _p(z), _p(y),
                                 _p(h_last), batch, L, D, N, _dtype_code(x), _stream(stream)),
           "ssm_conv_scan_fwd")


def ssm_scan_bwd(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last, du, ddelta, ddt_bias, dA,
                 dB, dC, dDskip, dz, stream=None) -> None:
    """Backward pass of ssm_scan_fwd: writes du, ddelta, dz (input dtype) and
    dB, dC, dA, ddt_bias, dDskip (float32) from dy (and dh_last, or None)."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_bwd(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip), _p(z),
                            _p(dy), _p(dh_last), _p(du), _p(ddelta), _p(ddt_bias), _p(dA), _p(dB),
                            _p(dC), _p(dDskip), _p(dz), batch, L, D, N, _dtype_code(u),
                            _stream(stream)), "ssm_scan_bwd")


def ssm_scan_fwd_ckpt(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, ckpt, stream=None) -> None:
    """ssm_scan_fwd that also writes ckpt [ceil(L/32), batch, D, 16] float32:
    the state entering every 32-step unit, for ssm_scan_bwd_ckpt."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_fwd_ckpt(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip),
                                 _p(z), _p(y), _p(h_last), _p(ckpt), batch, L, D, N,
                                 _dtype_code(u), _stream(stream)), "ssm_scan_fwd_ckpt")


def ssm_scan_bwd_ckpt(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last, ckpt, du, ddelta,
                      ddt_bias, dA, dB, dC, dDskip, dz, stream=None) -> None:
    """ssm_scan_bwd reading the unit states from ckpt (ssm_scan_fwd_ckpt's,
    same inputs) instead of recomputing them."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_bwd_ckpt(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip),
                                 _p(z), _p(dy), _p(dh_last), _p(ckpt), _p(du), _p(ddelta),
                                 _p(ddt_bias), _p(dA), _p(dB), _p(dC), _p(dDskip), _p(dz), batch,
                                 L, D, N, _dtype_code(u), _stream(stream)), "ssm_scan_bwd_ckpt")


def ssm_ssd_fwd(x, dt, dt_bias, A, B, C, Dskip, y, h_last, stream=None) -> None:
    """y, h_last <- the Mamba-2 (SSD) scan: x [Bt,L,H,P], dt [Bt,L,H], A [H],
    B/C [Bt,L,N]; h_last [Bt,H,P,N] float32 or None."""
    batch, L, H, P = x.shape
    N = B.shape[-1]
    _check(lib.ssm_ssd_fwd(_p(x), _p(dt), _p(dt_bias), _p(A), _p(B), _p(C), _p(Dskip), _p(y),
                           _p(h_last), batch, L, H, P, N, _dtype_code(x), _stream(stream)),
           "ssm_ssd_fwd")


def ssm_scan_fwd_noalloc(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, stream=None) -> None:
    """As ssm_scan_fwd, with the kernel scratch in the library's fixed device
    array instead of a stream-ordered allocation (for callers that cannot
    allocate device memory)."""
    batch, L, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_scan_fwd_noalloc(_p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C),
                                    _p(Dskip), _p(z), _p(y), _p(h_last), batch, L, D, N,
                                    _dtype_code(u), _stream(stream)), "ssm_scan_fwd_noalloc")


def ssm_step(state, u, delta, dt_bias, A, B, C, Dskip, z, y, stream=None) -> None:
    """state, y <- one decode step of (u, delta, dt_bias, A, B, C, Dskip, z)."""
    batch, D = u.shape
    N = A.shape[-1]
    _check(lib.ssm_step(_p(state), _p(u), _p(delta), _p(dt_bias), _p(A), _p(B), _p(C),
                        _p(Dskip), _p(z), _p(y), batch, D, N, _dtype_code(u),
                        _stream(stream)), "ssm_step")


def ssm_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device error status."""
    return lib.ssm_device_status(_stream(stream))


def ssm_abi_version() -> int:
    return lib.ssm_abi_version()


def ssm_unit_ceilings(reps: int = 5, stream=None) -> dict:
    """Measured unit rates of the current GPU (all SMs): fp32 multiply-adds/s
    (packed), special-function 2^x results/s, warp instructions issued/s."""
    out = (ctypes.c_double * 3)()
    _check(lib.ssm_unit_ceilings(out, int(reps), _stream(stream)), "ssm_unit_ceilings")
    return {"fma_per_s": out[0], "ex2_per_s": out[1], "warp_inst_per_s": out[2]}
