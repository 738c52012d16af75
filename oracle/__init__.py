"""FP64 CPU oracle for batch-invariant RMSNorm (TEST INFRASTRUCTURE ONLY).

Only the tests, the package smoke check and the bench's CPU-baseline leg
may import this package.  It shares no code with the CUDA library and never
imports it.  `rmsnorm_oracle.c` holds the arithmetic (plain FP64 loops);
this module compiles it with gcc and wraps it with ctypes.  `tree_replay`
holds an FP32 replay of the weight-gradient reduction order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics kept: no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                           "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_rmsnorm_fwd_f64.argtypes = [P, P, I, I, D, P, P]
        lib.oracle_rmsnorm_bwd_f64.argtypes = [P, P, P, I, I, D, P, P, P, P]
        lib.oracle_rmsnorm_fwd_bf16.argtypes = [P, P, I, I, D, P, P, P]
        lib.oracle_rmsnorm_bwd_bf16.argtypes = [P, P, P, I, I, D, P, P, P, P, P]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bit patterns."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(bits)


def forward_f64(x: np.ndarray, w: np.ndarray, eps: float):
    """(y, rstd) in float64 from float64 x [n,H], w [H]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    n, H = x.shape
    y = np.empty((n, H)); rstd = np.empty(n)
    _load().oracle_rmsnorm_fwd_f64(_ptr(x), _ptr(w), n, H, float(eps), _ptr(y), _ptr(rstd))
    return y, rstd


def backward_f64(x: np.ndarray, w: np.ndarray, dy: np.ndarray, eps: float):
    """(dx, dx_scale, dweight, dw_scale) in float64 from float64 inputs."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    n, H = x.shape
    dx = np.empty((n, H)); dxs = np.empty((n, H)); dw = np.empty(H); dws = np.empty(H)
    _load().oracle_rmsnorm_bwd_f64(_ptr(x), _ptr(w), _ptr(dy), n, H, float(eps),
                                   _ptr(dx), _ptr(dxs), _ptr(dw), _ptr(dws))
    return dx, dxs, dw, dws


def forward(x, w, eps: float):
    """(y, rstd) in float64 from bf16 x [n,H] (logical order, active rows only) and w [H]."""
    x = _u16(x); w = _u16(w)
    n, H = x.shape
    y = np.empty((n, H)); rstd = np.empty(n); scratch = np.empty(2 * H)
    _load().oracle_rmsnorm_fwd_bf16(_ptr(x), _ptr(w), n, H, float(eps), _ptr(y), _ptr(rstd),
                                    _ptr(scratch))
    return y, rstd


def backward(x, w, dy, eps: float, want_dx: bool = True):
    """(dx, dx_scale, dweight, dw_scale) in float64 from bf16 inputs in logical order.
    dx and dx_scale are None when want_dx is False (dweight only, O(H) memory)."""
    x = _u16(x); w = _u16(w); dy = _u16(dy)
    n, H = x.shape
    dx = np.empty((n, H)) if want_dx else None
    dxs = np.empty((n, H)) if want_dx else None
    dw = np.empty(H); dws = np.empty(H); scratch = np.empty(5 * H)
    _load().oracle_rmsnorm_bwd_bf16(_ptr(x), _ptr(w), _ptr(dy), n, H, float(eps),
                                    _ptr(dx), _ptr(dxs), _ptr(dw), _ptr(dws), _ptr(scratch))
    return dx, dxs, dw, dws
