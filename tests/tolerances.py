"""The one tolerance table of the test suite.

Invariance across layouts is bitwise (atol = 0, rtol = 0): compared on bit
patterns, never through this module.  Accuracy against the FP64 oracle uses:

* y (bf16):  |y - ref| <= max(2 ulp_bf16(ref), 1e-2 |ref|)
* dx (bf16): |dx - ref| <= max(2 ulp_bf16(ref), 1e-2 |ref|, 8 * 2^-24 * K)
             K = rstd * (|dy*w| + |xhat*m|) is the size of the two terms
             that cancel in dx; an FP32 evaluation of their difference is
             only accurate to a few 2^-24 of K, so where they cancel the
             result cannot be held to a bf16 ulp of the tiny difference.
* dweight (FP32): |dw - ref| <= 1e-4 * max(|ref|, S), S = sqrt(sum_g c_g^2)
             the root-sum-square of the column's terms c = dy*xhat; for a
             column whose sum nearly cancels, rounding noise is relative to
             S, not to the small sum.

ulp_bf16(v) is the spacing of bf16 numbers at |v| rounded to bf16 (2^-133
in the subnormal range).  The bare relative errors are reported alongside.
"""
from __future__ import annotations

import numpy as np

Y_ULPS = 2.0
Y_REL = 1e-2
DX_CANCEL = 8.0 * 2.0 ** -24
DW_REL = 1e-4


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(ref, dtype=np.float64))
    a = np.where(a < 2.0 ** -126, 2.0 ** -126, a)
    e = np.floor(np.log2(a))
    return np.where(a <= 2.0 ** -126, 2.0 ** -133, 2.0 ** (e - 7))


def bound_y(ref):
    ref = np.asarray(ref, dtype=np.float64)
    return np.maximum(Y_ULPS * ulp_bf16(ref), Y_REL * np.abs(ref))


def bound_dx(ref, k_scale):
    return np.maximum(bound_y(ref), DX_CANCEL * np.asarray(k_scale, dtype=np.float64))


def bound_dw(ref, s_scale):
    return DW_REL * np.maximum(np.abs(ref), np.asarray(s_scale, dtype=np.float64))


def check(name: str, got, ref, bound) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= bound)                       # NaN fails
    rel = err / np.maximum(np.abs(ref), 1e-30)
    out = {"tensor": name, "n": int(err.size), "violations": int(bad.sum()),
           "max_abs": float(np.nanmax(err)) if err.size else 0.0,
           "max_rel_bare": float(np.nanmax(rel)) if rel.size else 0.0,
           "max_err_over_bound": float(np.nanmax(err / bound)) if err.size else 0.0}
    if bad.any():
        i = int(np.flatnonzero(bad.reshape(-1))[0])
        out["first"] = {"index": i, "got": float(got.reshape(-1)[i]), "ref": float(ref.reshape(-1)[i]),
                        "bound": float(np.broadcast_to(bound, ref.shape).reshape(-1)[i])}
    return out
