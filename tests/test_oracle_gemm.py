"""Pins of the weight-gradient oracle of a linear layer (CPU)."""
import numpy as np
import pytest

from oracle import gemm


def test_hand_worked_case():
    x = np.array([[1.0, 2.0], [3.0, 4.0]])
    dy = np.array([[1.0, 0.0], [0.0, 2.0]])
    dw, s = gemm.dw_f64(x, dy)
    assert np.array_equal(dw, np.array([[1.0, 2.0], [6.0, 8.0]]))    # dy^T x by hand
    assert np.allclose(s, np.array([[1.0, 2.0], [6.0, 8.0]]))        # one term per entry


@pytest.mark.parametrize("scale", [1.0, 0.25])
def test_matches_finite_differences(scale):
    rng = np.random.default_rng(4)
    n, i, o = 5, 3, 4
    x, dy, w = rng.normal(size=(n, i)), rng.normal(size=(n, o)), rng.normal(size=(o, i))

    def loss(w_):
        return scale * np.sum(dy * (x @ w_.T))

    dw, _ = gemm.dw_f64(x, dy, scale)
    h = 1e-6
    for a in range(o):
        for b in range(i):
            e = np.zeros_like(w)
            e[a, b] = h
            g = (loss(w + e) - loss(w - e)) / (2 * h)
            assert abs(g - dw[a, b]) <= 1e-7 * max(1.0, abs(dw[a, b]))


def test_bf16_entry_widens_exactly():
    rng = np.random.default_rng(5)
    xb = (rng.integers(0, 1 << 16, size=(4, 8), dtype=np.uint32) & 0x7F7F).astype(np.uint16)
    db = (rng.integers(0, 1 << 16, size=(4, 8), dtype=np.uint32) & 0x3F7F).astype(np.uint16)
    d1, _ = gemm.dw(xb, db)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    df = (db.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(d1, df.T @ xf)
