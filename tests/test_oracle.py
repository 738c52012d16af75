"""Pins of the FP64 oracle against facts other than its own formula.

Hand-worked examples (tests/golden/hand_examples.json), closed forms of
special cases, invariants of the method and central finite differences.
Each check is chosen so that a plausible slip in the oracle (eps outside the
root, sum instead of mean, a dropped term or wrong sign in dx, dweight
without the normalisation, a transposed operand) fails at least one.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(v):
    """bf16 bit patterns of values that are exactly representable in bf16."""
    f = np.asarray(v, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def test_bf16_widening_known_patterns():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x4B80) == 16777216.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133          # smallest subnormal
    assert oracle.bf16_to_double(0x7F80) == float("inf")
    assert np.isnan(oracle.bf16_to_double(0x7FC0))
    assert np.signbit(oracle.bf16_to_double(0x8000))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "hand_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    x = _bf16_bits(case["x"]); w = _bf16_bits(case["w"]); dy = _bf16_bits(case["dy"])
    y, rstd = oracle.forward(x, w, case["eps"])
    np.testing.assert_allclose(y, case["y"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(rstd, case["rstd"], rtol=1e-14)
    dx, _, dw, _ = oracle.backward(x, w, dy, case["eps"])
    np.testing.assert_allclose(dx, case["dx"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dw, case["dweight"], rtol=1e-13, atol=1e-15)


def test_constant_row_maps_to_w_times_sign():
    rng = np.random.default_rng(1)
    H = 16
    w = rng.normal(size=H)
    for c in (-3.0, 0.125, 7.5, -1e3):
        x = np.full((1, H), c)
        y, _ = oracle.forward_f64(x, w, 0.0)
        np.testing.assert_allclose(y[0], w * np.sign(c), rtol=1e-15)
        y, _ = oracle.forward_f64(x, w, 1e-6)                  # eps perturbs below 1e-6/c^2
        np.testing.assert_allclose(y[0], w * np.sign(c), rtol=1e-6 / c ** 2 + 1e-15)


def test_scale_invariance_and_unit_rms_at_zero_eps():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(5, 24)); w = rng.normal(size=24) + 2.0
    y1, r1 = oracle.forward_f64(x, w, 0.0)
    y2, r2 = oracle.forward_f64(3.5 * x, w, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    np.testing.assert_allclose(r1, 3.5 * r2, rtol=1e-13)
    xhat = y1 / w
    np.testing.assert_allclose(np.mean(xhat ** 2, axis=1), 1.0, rtol=1e-13)   # mean, not sum


def test_small_input_limit_pins_eps_placement():
    # |x| << sqrt(eps): y -> x*w/sqrt(eps) (eps added to the mean, inside the root)
    x = np.array([[1e-6, -2e-6, 3e-6, 0.5e-6]]); w = np.array([1.0, 2.0, -1.0, 4.0])
    y, _ = oracle.forward_f64(x, w, 4.0)
    np.testing.assert_allclose(y[0], x[0] * w / 2.0, rtol=1e-11)
    y0, r0 = oracle.forward_f64(np.zeros((1, 4)), w, 1e-6)     # zero row stays finite
    assert np.all(y0 == 0) and np.isclose(r0[0], 1e3)


def _loss(x, w, dy, eps):
    y, _ = oracle.forward_f64(x, w, eps)
    return float(np.sum(dy * y))


@pytest.mark.parametrize("H", [1, 3, 4, 8])
def test_dx_and_dweight_match_central_finite_differences(H):
    rng = np.random.default_rng(10 + H)
    n, eps, step = 3, 1e-3, 1e-5
    x = rng.normal(size=(n, H)); w = 1 + 0.1 * rng.normal(size=H); dy = rng.normal(size=(n, H))
    dx, _, dw, _ = oracle.backward_f64(x, w, dy, eps)
    fd_dx = np.zeros_like(x)
    for g in range(n):
        for h in range(H):
            xp = x.copy(); xp[g, h] += step
            xm = x.copy(); xm[g, h] -= step
            fd_dx[g, h] = (_loss(xp, w, dy, eps) - _loss(xm, w, dy, eps)) / (2 * step)
    fd_dw = np.zeros(H)
    for h in range(H):
        wp = w.copy(); wp[h] += step
        wm = w.copy(); wm[h] -= step
        fd_dw[h] = (_loss(x, wp, dy, eps) - _loss(x, wm, dy, eps)) / (2 * step)
    np.testing.assert_allclose(dx, fd_dx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dw, fd_dw, rtol=1e-6, atol=1e-8)


def test_h1_closed_form():
    x = np.array([[0.3], [-2.0], [5.0]]); w = np.array([1.7]); dy = np.array([[1.0], [-0.5], [2.0]])
    eps = 0.25
    dx, _, dw, _ = oracle.backward_f64(x, w, dy, eps)
    expect = dy * w * eps / (x ** 2 + eps) ** 1.5
    np.testing.assert_allclose(dx, expect, rtol=1e-13)
    np.testing.assert_allclose(dw, [np.sum(dy[:, 0] * x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps))], rtol=1e-13)


def test_dx_orthogonality_invariant():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(4, 32)); w = rng.normal(size=32); dy = rng.normal(size=(4, 32))
    dx0, _, _, _ = oracle.backward_f64(x, w, dy, 0.0)
    np.testing.assert_allclose(np.sum(dx0 * x, axis=1), 0.0, atol=1e-12)
    eps = 0.7
    dx, _, _, _ = oracle.backward_f64(x, w, dy, eps)
    ms = np.mean(x ** 2, axis=1); rstd = 1 / np.sqrt(ms + eps)
    gx = np.sum(dy * w * x, axis=1)
    np.testing.assert_allclose(np.sum(dx * x, axis=1), rstd * gx * eps / (ms + eps), rtol=1e-11)


def test_dweight_exact_integer_case():
    # eps=0, rows of +-2^k: xhat = +-1 exactly, so dweight is an exact integer sum
    H = 8
    signs = np.array([1, -1, 1, 1, -1, -1, 1, -1], dtype=np.float64)
    x = np.stack([signs * 4.0, -signs * 0.5, signs * 2.0])
    dy = np.array([[1, 2, 3, 4, 5, 6, 7, 8], [-1, 0, 2, 0, 1, 1, 1, 3], [9, 9, 9, 9, 9, 9, 9, 9]], dtype=np.float64)
    w = np.ones(H)
    _, _, dw, dws = oracle.backward_f64(x, w, dy, 0.0)
    expect = dy[0] * signs - dy[1] * signs + dy[2] * signs
    assert np.array_equal(dw, expect)
    assert np.allclose(dws, np.sqrt(np.sum(dy ** 2, axis=0)))


def test_bf16_and_f64_entry_points_agree():
    rng = np.random.default_rng(4)
    xf = rng.normal(size=(6, 40)).astype(np.float32); wf = (1 + 0.1 * rng.normal(size=40)).astype(np.float32)
    dyf = rng.normal(size=(6, 40)).astype(np.float32)
    def tobits(a):
        return (a.view(np.uint32) >> 16).astype(np.uint16)
    xb, wb, dyb = tobits(xf), tobits(wf), tobits(dyf)
    def back(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y1, r1 = oracle.forward(xb, wb, 1e-6)
    y2, r2 = oracle.forward_f64(back(xb), back(wb), 1e-6)
    assert np.array_equal(y1, y2) and np.array_equal(r1, r2)
    a = oracle.backward(xb, wb, dyb, 1e-6)
    b = oracle.backward_f64(back(xb), back(wb), back(dyb), 1e-6)
    for u, v in zip(a, b):
        np.testing.assert_allclose(u, v, rtol=1e-15, atol=0)
    _, _, dw_only, dws_only = oracle.backward(xb, wb, dyb, 1e-6, want_dx=False)
    assert np.array_equal(dw_only, a[2]) and np.array_equal(dws_only, a[3])
