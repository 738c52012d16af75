"""FP64 oracle of the norm's neighbours in a training chain (TEST INFRASTRUCTURE ONLY).

Two steps sit on either side of RMSNorm when it runs inside a model
("[WS1 Closeout][Backward] ..." issue #270, "Scope": the upstream gradient,
the loss reduction and the active-token denominator are fixed across
configurations; "WS1 C4 (#270) closeout evidence", "Acceptance map": the
harness injects the active-token denominator and seeds the backward with an
upstream that depends on logical identity only):

* the residual add in front of the norm, h = x + r, where h also continues
  along the residual stream and is stored in bf16;
* the loss seed behind it: a mean over the D active tokens of the whole
  multiset scales every upstream gradient by 1/D.

Plain definitions, evaluated in float64:

    h      = round_bf16(x + r)                  (the stored residual stream)
    y      = h * w / sqrt(mean(h^2) + eps)      (the norm of h)
    dh     = s * dx_norm(h, dy) + dres          (s = grad_scale = 1/D)
    dweight= s * sum_rows dy * h * rstd(h)

dres is the gradient reaching h along the residual path.  The sums over rows
and columns are the FP64 loops of rmsnorm_oracle.c; nothing here is blocked
or reordered.  Pins: `round_bf16` against PyTorch's float32-to-bfloat16
conversion (round to nearest even) and hand-made ties; the backward against
central finite differences of the scalar L = s * sum(dy * y) + sum(dres * h).
"""
from __future__ import annotations

import numpy as np

from . import _u16, backward, backward_f64, forward_f64


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of a binary32)."""
    b = np.asarray(_u16(bits), dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_bf16(v) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest, ties to even.

    bf16 keeps 8 significant bits (7 stored) and the exponent range of
    binary32: normal numbers from 2^-126, subnormals in steps of 2^-133,
    overflow to infinity at (2 - 2^-8) * 2^127 and above."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    m, e = np.frexp(a)                                   # a = m * 2^e, m in [0.5, 1)
    q = np.maximum(e - 1, -126) - 7                     # exponent of the spacing at a
    n = np.rint(np.ldexp(a, -q))                        # multiples of the spacing, ties to even
    r = np.ldexp(n, q)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.where(np.isinf(a), np.inf, r)
    out = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out = np.where(np.signbit(v), out | np.uint16(0x8000), out)
    out = np.where(np.isnan(v), np.uint16(0x7FC0), out)
    return out.astype(np.uint16)


def add_forward_f64(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float, round_h: bool = True):
    """(h, y, rstd) in float64; h rounded to bf16 unless round_h is False."""
    s = np.asarray(x, dtype=np.float64) + np.asarray(r, dtype=np.float64)
    h = bf16_bits_to_f64(round_bf16(s)) if round_h else s
    y, rstd = forward_f64(h, w, eps)
    return h, y, rstd


def add_forward(x, r, w, eps: float):
    """(h_bits, y, rstd) from bf16 x, r [n, H] and w [H] in logical order."""
    x64, r64 = bf16_bits_to_f64(x), bf16_bits_to_f64(r)
    h_bits = round_bf16(x64 + r64)
    y, rstd = forward_f64(bf16_bits_to_f64(h_bits), bf16_bits_to_f64(w), eps)
    return h_bits, y, rstd


def add_backward_f64(h: np.ndarray, w: np.ndarray, dy: np.ndarray, dres, eps: float, grad_scale: float):
    """(dh, dh_scale, dweight, dw_scale) in float64 from float64 inputs.

    dh_scale = s*K + |dres| is the size of the terms that meet in dh (K the
    norm backward's own cancellation scale); dw_scale = |s| * S."""
    dx, k, dw, sc = backward_f64(h, w, dy, eps)
    s = float(grad_scale)
    dres = np.zeros_like(dx) if dres is None else np.asarray(dres, dtype=np.float64)
    return s * dx + dres, abs(s) * k + np.abs(dres), s * dw, abs(s) * sc


def add_backward(h, w, dy, dres, eps: float, grad_scale: float, want_dx: bool = True):
    """(dh, dh_scale, dweight, dw_scale) from bf16 inputs in logical order;
    dh and dh_scale are None when want_dx is False."""
    dx, k, dw, sc = backward(h, w, dy, eps, want_dx=want_dx)
    s = float(grad_scale)
    if want_dx:
        d = np.zeros_like(dx) if dres is None else bf16_bits_to_f64(dres)
        return s * dx + d, abs(s) * k + np.abs(d), s * dw, abs(s) * sc
    return None, None, s * dw, abs(s) * sc
