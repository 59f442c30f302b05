"""float64 CPU oracle for the selective state-space scan (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may load it.  It shares no code with the CUDA library in
``selective_state_space_113_b300``; the two meet only in the seeded input
generators of ``selective_state_space_113_b300.workloads``, which hold none of
the method's arithmetic.

The arithmetic lives in ``ssm_oracle.c`` (plain C, float64, sequential in t);
this module compiles it with gcc and calls it through ctypes.  ctypes releases
the GIL during the call, so independent channel ranges run on a thread pool.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ssm_oracle.c")
LIB = os.path.join(HERE, "libssmoracle.so")

_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_scan_fwd.restype = ctypes.c_int
    lib.oracle_scan_fwd.argtypes = [vp] * 10 + [i64] * 4 + [ctypes.c_int, i64, i64]
    lib.oracle_step.restype = ctypes.c_int
    lib.oracle_step.argtypes = [vp] * 10 + [i64] * 3 + [ctypes.c_int]
    lib.oracle_scan_fwd_disc.restype = ctypes.c_int
    lib.oracle_scan_fwd_disc.argtypes = [vp] * 10 + [i64] * 4 + [ctypes.c_int, ctypes.c_int,
                                                                 i64, i64]
    lib.oracle_conv_scan_fwd.restype = ctypes.c_int
    lib.oracle_conv_scan_fwd.argtypes = ([vp] * 3 + [ctypes.c_int] + [vp] * 9 + [i64] * 4
                                         + [ctypes.c_int, i64, i64])
    lib.oracle_scan_bwd.restype = ctypes.c_int
    lib.oracle_scan_bwd.argtypes = [vp] * 18 + [i64] * 4 + [ctypes.c_int, i64, i64]
    lib.oracle_abi_version.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) an oracle library.

    With ``path`` given, loads that build (the planted-mistake tests use
    this); otherwise the cached default build next to this file.
    """
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(LIB)
                    or os.path.getmtime(LIB) < os.path.getmtime(SRC)):
                build()
            lib = _bind(ctypes.CDLL(LIB))
            if lib.oracle_abi_version() != 4:
                raise RuntimeError("stale oracle build: " + LIB)
            _lib = lib
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_input(a, dtype: int):
    """Return a C-contiguous numpy view of an input tensor in the oracle's dtype.

    float32 inputs stay float32; bfloat16 inputs must arrive as uint16 bit
    patterns (see ``bits_of``).
    """
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = np.float32 if dtype == F32 else np.uint16
    if a.dtype != want:
        raise TypeError(f"expected {want.__name__} input, got {a.dtype}")
    return a


def _as_f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def bits_of(t) -> np.ndarray:
    """Host numpy array of a torch tensor: float32 as is, bf16 as uint16 bits."""
    import torch
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")


def scan_fwd(u, delta, dt_bias, A, B, C, Dskip, z, dtype: int = F32,
             threads: int = 1, lib: ctypes.CDLL | None = None):
    """Selective scan, float64.  Shapes: u/delta/z [Bt,L,D], B/C [Bt,L,N], A [D,N].

    Returns ``(y [Bt,L,D] float64, h_last [Bt,D,N] float64)``.
    """
    lib = lib or load()
    u, delta, z = (_as_input(x, dtype) for x in (u, delta, z))
    B, C = _as_input(B, dtype), _as_input(C, dtype)
    A, dt_bias, Dskip = _as_f32(A), _as_f32(dt_bias), _as_f32(Dskip)
    batch, L, D = u.shape
    N = A.shape[1]
    if A.shape != (D, N) or B.shape != (batch, L, N) or C.shape != (batch, L, N):
        raise ValueError("inconsistent shapes")
    y = np.zeros((batch, L, D), np.float64)
    h = np.zeros((batch, D, N), np.float64)
    threads = max(1, min(int(threads), D)) if D else 1

    def run(lo, hi):
        rc = lib.oracle_scan_fwd(_ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A),
                                 _ptr(B), _ptr(C), _ptr(Dskip), _ptr(z),
                                 _ptr(y), _ptr(h), batch, L, D, N, dtype, lo, hi)
        if rc != 0:
            raise RuntimeError(f"oracle_scan_fwd returned {rc}")

    if threads == 1:
        run(0, D)
    else:
        bounds = np.linspace(0, D, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])),
                        range(threads)))
    return y, h


ZOH, EULER, TRAPEZOID = 0, 1, 2


def scan_fwd_disc(u, delta, dt_bias, A, B, C, Dskip, z, disc: int, dtype: int = F32,
                  threads: int = 1, lib: ctypes.CDLL | None = None):
    """Selective scan with a discretisation variant (ZOH, EULER or TRAPEZOID),
    float64; arguments and results as for ``scan_fwd``."""
    lib = lib or load()
    u, delta, z = (_as_input(x, dtype) for x in (u, delta, z))
    B, C = _as_input(B, dtype), _as_input(C, dtype)
    A, dt_bias, Dskip = _as_f32(A), _as_f32(dt_bias), _as_f32(Dskip)
    batch, L, D = u.shape
    N = A.shape[1]
    if A.shape != (D, N) or B.shape != (batch, L, N) or C.shape != (batch, L, N):
        raise ValueError("inconsistent shapes")
    y = np.zeros((batch, L, D), np.float64)
    h = np.zeros((batch, D, N), np.float64)
    threads = max(1, min(int(threads), D)) if D else 1

    def run(lo, hi):
        rc = lib.oracle_scan_fwd_disc(_ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A),
                                      _ptr(B), _ptr(C), _ptr(Dskip), _ptr(z),
                                      _ptr(y), _ptr(h), batch, L, D, N, dtype, int(disc), lo, hi)
        if rc != 0:
            raise RuntimeError(f"oracle_scan_fwd_disc returned {rc}")

    if threads == 1:
        run(0, D)
    else:
        bounds = np.linspace(0, D, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])),
                        range(threads)))
    return y, h


def conv_scan_fwd(x, conv_w, conv_b, act, delta, dt_bias, A, B, C, Dskip, z,
                  dtype: int = F32, threads: int = 1, lib: ctypes.CDLL | None = None):
    """Causal depthwise width-4 convolution of x (conv_w [D,4] float32, conv_b
    [D] or None; act 1 applies SiLU) feeding the zero-order-hold scan, float64.
    Returns ``(y, h_last)`` as ``scan_fwd``."""
    lib = lib or load()
    x, delta, z = (_as_input(v, dtype) for v in (x, delta, z))
    B, C = _as_input(B, dtype), _as_input(C, dtype)
    A, dt_bias, Dskip = _as_f32(A), _as_f32(dt_bias), _as_f32(Dskip)
    conv_w, conv_b = _as_f32(conv_w), _as_f32(conv_b)
    batch, L, D = x.shape
    N = A.shape[1]
    if A.shape != (D, N) or B.shape != (batch, L, N) or conv_w.shape != (D, 4):
        raise ValueError("inconsistent shapes")
    y = np.zeros((batch, L, D), np.float64)
    h = np.zeros((batch, D, N), np.float64)
    threads = max(1, min(int(threads), D)) if D else 1

    def run(lo, hi):
        rc = lib.oracle_conv_scan_fwd(_ptr(x), _ptr(conv_w), _ptr(conv_b), int(act), _ptr(delta),
                                      _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                                      _ptr(z), _ptr(y), _ptr(h), batch, L, D, N, dtype, lo, hi)
        if rc != 0:
            raise RuntimeError(f"oracle_conv_scan_fwd returned {rc}")

    if threads == 1:
        run(0, D)
    else:
        bounds = np.linspace(0, D, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])),
                        range(threads)))
    return y, h


def scan_bwd(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last=None, dtype: int = F32,
             threads: int = 1, lib: ctypes.CDLL | None = None):
    """Backward pass of the zero-order-hold scan, float64: the derivatives of a
    loss with dLoss/dy = dy ([Bt,L,D], the input dtype) and dLoss/dh_last =
    dh_last ([Bt,D,N] float32, None = 0).

    Returns a dict of float64 arrays: du, ddelta, dz ([Bt,L,D]; dz None
    without z), dB, dC ([Bt,L,N]), dA ([D,N]), ddt_bias, dDskip ([D]).
    """
    lib = lib or load()
    u, delta, z, dy = (_as_input(x, dtype) for x in (u, delta, z, dy))
    B, C = _as_input(B, dtype), _as_input(C, dtype)
    A, dt_bias, Dskip = _as_f32(A), _as_f32(dt_bias), _as_f32(Dskip)
    dh_last = _as_f32(dh_last)
    batch, L, D = u.shape
    N = A.shape[1]
    if (A.shape != (D, N) or B.shape != (batch, L, N) or C.shape != (batch, L, N)
            or dy.shape != u.shape or (dh_last is not None and dh_last.shape != (batch, D, N))):
        raise ValueError("inconsistent shapes")
    du = np.zeros((batch, L, D), np.float64)
    ddelta = np.zeros((batch, L, D), np.float64)
    dz = np.zeros((batch, L, D), np.float64) if z is not None else None
    dA = np.zeros((D, N), np.float64)
    ddt_bias = np.zeros(D, np.float64)
    dDskip = np.zeros(D, np.float64)
    threads = max(1, min(int(threads), D)) if D else 1
    parts = [(np.zeros((batch, L, N)), np.zeros((batch, L, N))) for _ in range(threads)]

    def run(i, lo, hi):
        dB_i, dC_i = parts[i]
        rc = lib.oracle_scan_bwd(_ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(Dskip), _ptr(z), _ptr(dy), _ptr(dh_last), _ptr(du),
                                 _ptr(ddelta), _ptr(ddt_bias), _ptr(dA), _ptr(dB_i), _ptr(dC_i),
                                 _ptr(dDskip), _ptr(dz), batch, L, D, N, dtype, lo, hi)
        if rc != 0:
            raise RuntimeError(f"oracle_scan_bwd returned {rc}")

    bounds = np.linspace(0, D, threads + 1).astype(np.int64)
    if threads == 1:
        run(0, 0, D)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(i, int(bounds[i]), int(bounds[i + 1])), range(threads)))
    dB = sum(p[0] for p in parts)
    dC = sum(p[1] for p in parts)
    return dict(du=du, ddelta=ddelta, dz=dz, dB=dB, dC=dC, dA=dA, ddt_bias=ddt_bias,
                dDskip=dDskip)


def ssd_fwd(x, dt, dt_bias, A, B, C, Dskip, dtype: int = F32, threads: int = 1,
            lib: ctypes.CDLL | None = None):
    """The Mamba-2 form of the scan (structured state-space duality), float64:
    one scalar A per head, the input term dt B x (Euler), head dimension P.

    x [Bt,L,H,P], dt [Bt,L,H] (before softplus), B/C [Bt,L,N] (input dtype);
    dt_bias [H], A [H], Dskip [H] (float32, dt_bias/Dskip may be None).
    For channel (h, p) this is exactly the Euler scan with A[d, n] = A[h] for
    every n, delta[b, t, d] = dt[b, t, h], dt_bias[d] = dt_bias[h] and
    Dskip[d] = Dskip[h], without a gate; the oracle is that scan, on channels
    numbered d = h P + p.  Returns (y [Bt,L,H,P], h_last [Bt,H,P,N]).
    """
    x = np.ascontiguousarray(x)
    dt = np.ascontiguousarray(dt)
    batch, L, H, P = x.shape
    N = B.shape[-1]
    if dt.shape != (batch, L, H) or B.shape != (batch, L, N) or C.shape != (batch, L, N):
        raise ValueError("inconsistent shapes")
    u = x.reshape(batch, L, H * P)
    delta = np.ascontiguousarray(np.repeat(dt, P, axis=2))
    Ad = np.ascontiguousarray(np.repeat(np.asarray(A, np.float32), P)[:, None] * np.ones(N, np.float32))
    bias = None if dt_bias is None else np.repeat(np.asarray(dt_bias, np.float32), P)
    skip = None if Dskip is None else np.repeat(np.asarray(Dskip, np.float32), P)
    y, h = scan_fwd_disc(u, delta, bias, Ad, B, C, skip, None, EULER, dtype=dtype,
                         threads=threads, lib=lib)
    return y.reshape(batch, L, H, P), h.reshape(batch, H, P, N)


def step(state, u, delta, dt_bias, A, B, C, Dskip, z, dtype: int = F32,
         lib: ctypes.CDLL | None = None):
    """One decode step, float64.  state [Bt,D,N] (copied), u/delta/z [Bt,D], B/C [Bt,N].

    Returns ``(new_state, y [Bt,D])``.
    """
    lib = lib or load()
    u, delta, z = (_as_input(x, dtype) for x in (u, delta, z))
    B, C = _as_input(B, dtype), _as_input(C, dtype)
    A, dt_bias, Dskip = _as_f32(A), _as_f32(dt_bias), _as_f32(Dskip)
    st = np.array(state, dtype=np.float64, order="C", copy=True)
    batch, D = u.shape
    N = A.shape[1]
    if st.shape != (batch, D, N) or B.shape != (batch, N):
        raise ValueError("inconsistent shapes")
    y = np.zeros((batch, D), np.float64)
    rc = lib.oracle_step(_ptr(st), _ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A),
                         _ptr(B), _ptr(C), _ptr(Dskip), _ptr(z), _ptr(y),
                         batch, D, N, dtype)
    if rc != 0:
        raise RuntimeError(f"oracle_step returned {rc}")
    return st, y
