"""FP64 oracle of the linear layer's weight gradient (TEST INFRASTRUCTURE ONLY).

For y = x W^T over the logical tokens g of a multiset, the weight gradient is
dW = sum_g dy_g^T x_g, i.e. dW[o][i] = sum_g dy[g][o] * x[g][i] ("WS1 C4 (#270)
closeout evidence": det_gemm's dW is the weight gradient that failed the
chunk and singleton checks).  Evaluated in float64 from the bf16 inputs (a
library matrix product as the one step), with the scale of the terms for
the tolerance: S[o][i] = sqrt(sum_g (dy[g][o] * x[g][i])^2).  Pins: central
finite differences of L(W) = sum(dy * (x W^T)) and a hand-worked 2 x 2 case.
"""
from __future__ import annotations

import numpy as np

from . import _u16


def _f64(bits) -> np.ndarray:
    b = np.asarray(_u16(bits), dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def dw_f64(x: np.ndarray, dy: np.ndarray, grad_scale: float = 1.0):
    """(dW [O][I], S [O][I]) in float64 from float64 x [N][I], dy [N][O]."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    dw = float(grad_scale) * (dy.T @ x)
    s = abs(float(grad_scale)) * np.sqrt((dy * dy).T @ (x * x))
    return dw, s


def dw(x_bits, dy_bits, grad_scale: float = 1.0):
    """(dW, S) from bf16 x [N][I] and dy [N][O] in logical order."""
    return dw_f64(_f64(x_bits), _f64(dy_bits), grad_scale)
