"""Pins of the chain oracle (residual add, loss seed) against facts outside it (CPU)."""
import numpy as np
import pytest
import torch

from oracle import chain


def _torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_round_bf16_matches_torch_conversion_on_binary32_values():
    """PyTorch's float32 -> bfloat16 cast rounds to nearest even; on values that
    are exact in binary32 it is the correctly rounded result."""
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    # ties: low 16 bits exactly 0x8000, with even and odd kept parts
    t = (rng.integers(0, 2 ** 16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    t = t.view(np.float32)
    t = t[np.isfinite(t)]
    for arr in (v, t, np.array([0.0, -0.0, 1e-45, -1e-45, 3.4e38, -3.4e38], np.float32)):
        got = chain.round_bf16(arr.astype(np.float64))
        want = _torch_bf16_bits(arr)
        assert np.array_equal(got, want), np.flatnonzero(got != want)[:5]


def test_round_bf16_hand_cases():
    one = 0x3F80
    assert chain.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == one                  # tie -> even (1.0)
    assert chain.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == one + 2          # tie -> even (1 + 2^-6)
    assert chain.round_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == one + 1  # above the tie: up
    assert chain.round_bf16(np.array([2.0 ** -133]))[0] == 0x0001                   # smallest subnormal
    assert chain.round_bf16(np.array([2.0 ** -134]))[0] == 0x0000                   # tie -> even (0)
    assert chain.round_bf16(np.array([(2 - 2.0 ** -8) * 2.0 ** 127]))[0] == 0x7F80  # overflow to inf
    assert chain.round_bf16(np.array([(2 - 2.0 ** -7) * 2.0 ** 127]))[0] == 0x7F7F  # largest finite
    assert chain.round_bf16(np.array([-0.0]))[0] == 0x8000
    assert chain.round_bf16(np.array([np.nan]))[0] & 0x7F80 == 0x7F80


def test_add_forward_special_cases():
    rng = np.random.default_rng(1)
    x = chain.round_bf16(rng.normal(size=(5, 16)))
    zero = np.zeros_like(x)
    w = chain.round_bf16(1 + 0.1 * rng.normal(size=16))
    h, y, _ = chain.add_forward(x, zero, w, 1e-6)
    assert np.array_equal(h, x)                              # r = 0: h is x, bit for bit
    # small integers: the sum is exact, so h is the sum itself
    xi = chain.round_bf16(rng.integers(-100, 100, size=(3, 8)).astype(np.float64))
    ri = chain.round_bf16(rng.integers(-100, 100, size=(3, 8)).astype(np.float64))
    h2, _, _ = chain.add_forward(xi, ri, w[:8], 1e-6)
    assert np.array_equal(chain.bf16_bits_to_f64(h2), chain.bf16_bits_to_f64(xi) + chain.bf16_bits_to_f64(ri))
    # y follows the closed form of the norm of h
    hf = chain.bf16_bits_to_f64(h)
    want = hf * chain.bf16_bits_to_f64(w) / np.sqrt((hf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(y, want, rtol=1e-13)


@pytest.mark.parametrize("H", [1, 4, 8])
@pytest.mark.parametrize("s", [1.0, 1.0 / 3.0, 2.0 ** -10])
def test_add_backward_matches_finite_differences(H, s):
    """L(x, r, w) = s * sum(dy * y(x + r)) + sum(dres * (x + r)), h unrounded."""
    rng = np.random.default_rng(H * 7 + int(1 / s))
    n, eps = 3, 1e-3
    x, r = rng.normal(size=(n, H)), rng.normal(size=(n, H))
    w = 1 + 0.1 * rng.normal(size=H)
    dy, dres = rng.normal(size=(n, H)), rng.normal(size=(n, H))

    def L(x_, r_, w_):
        _, y, _ = chain.add_forward_f64(x_, r_, w_, eps, round_h=False)
        return s * np.sum(dy * y) + np.sum(dres * (x_ + r_))

    dh, _, dw, _ = chain.add_backward_f64(x + r, w, dy, dres, eps, s)
    step = 1e-6
    for i in range(n):
        for j in range(H):
            e = np.zeros((n, H)); e[i, j] = step
            gx = (L(x + e, r, w) - L(x - e, r, w)) / (2 * step)
            gr = (L(x, r + e, w) - L(x, r - e, w)) / (2 * step)
            assert abs(gx - dh[i, j]) <= 1e-6 * max(1.0, abs(dh[i, j]))
            assert abs(gr - dh[i, j]) <= 1e-6 * max(1.0, abs(dh[i, j]))
    for j in range(H):
        e = np.zeros(H); e[j] = step
        g = (L(x, r, w + e) - L(x, r, w - e)) / (2 * step)
        assert abs(g - dw[j]) <= 1e-6 * max(1.0, abs(dw[j]))


def test_add_backward_bf16_entry_agrees_with_f64_entry():
    rng = np.random.default_rng(3)
    h = chain.round_bf16(rng.normal(size=(6, 24)))
    w = chain.round_bf16(1 + 0.1 * rng.normal(size=24))
    dy = chain.round_bf16(rng.normal(size=(6, 24)) * 1e-2)
    dres = chain.round_bf16(rng.normal(size=(6, 24)) * 1e-2)
    a = chain.add_backward(h, w, dy, dres, 1e-6, 0.125)
    b = chain.add_backward_f64(chain.bf16_bits_to_f64(h), chain.bf16_bits_to_f64(w), chain.bf16_bits_to_f64(dy),
                               chain.bf16_bits_to_f64(dres), 1e-6, 0.125)
    for u, v in zip(a, b):
        np.testing.assert_allclose(u, v, rtol=1e-14, atol=0)
