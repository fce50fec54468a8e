"""Pins of the oracle's residual add + RMS norm + weight multiply (the
fusion the lucebox commit list describes for the steps around a block: the
residual sum is kept beside the normalised output).  Each check is a closed
form or an invariance the definition implies, not a retyped formula."""
import numpy as np
import pytest

import oracle
import workloads as W


def bf16(v):
    return W.f32_to_bf16_bits(np.asarray(v, np.float32))


def f(b):
    return W.bf16_bits_to_f32(np.asarray(b, np.uint16)).astype(np.float64)


def gamma(H, seed=3):
    return W.bf16_normal((H,), W.stream_key(seed, "misc"), 1.0)


@pytest.mark.parametrize("c", [3.0, -0.5, 1024.0])
def test_constant_rows_normalise_to_plus_or_minus_gamma(c):
    H = 128
    g = gamma(H)
    resid = np.tile(bf16([c] * H), (2, 1))
    r_out, x = oracle.add_rmsnorm(resid, np.zeros((2, H)), g, 0.0)
    assert np.array_equal(r_out, resid)
    assert np.array_equal(f(x[0]), np.sign(c) * f(g))


def test_eps_enters_under_the_root():
    # 3 / sqrt(3^2 + 7) = 3/4 exactly
    H = 64
    r_out, x = oracle.add_rmsnorm(np.tile(bf16([3.0] * H), (1, 1)), np.zeros((1, H)),
                                  bf16([1.0] * H), 7.0)
    assert (f(x) == 0.75).all()


def test_one_hot_row_scales_by_root_H():
    H = 256  # sqrt(H) = 16: the normalised one-hot entry is 16 * sign(a)
    g = gamma(H, seed=5)
    for j, a in ((0, 2.5), (17, -0.125), (255, 96.0)):
        resid = np.zeros((1, H), np.uint16)
        resid[0, j] = bf16([a])[0]
        _, x = oracle.add_rmsnorm(resid, np.zeros((1, H)), g, 0.0)
        want = np.zeros(H)
        want[j] = 16.0 * np.sign(a) * f(g)[j]
        assert np.array_equal(f(x[0]), f(bf16(want)))


def test_scaling_the_residual_by_a_power_of_two_leaves_x_next_unchanged():
    H = 512
    g = gamma(H, seed=7)
    base = W.bf16_normal((2, H), W.stream_key(8, "misc"), 1.0)
    _, x0 = oracle.add_rmsnorm(base, np.zeros((2, H)), g, 0.0)
    for k in (-6, -1, 3, 9):
        scaled = bf16(f(base) * 2.0 ** k)  # exact in bf16
        _, xk = oracle.add_rmsnorm(scaled, np.zeros((2, H)), g, 0.0)
        assert np.array_equal(xk, x0)


@pytest.mark.parametrize("resid,block,want", [
    (1.0, 2.0 ** -8, 1.0),                      # half an ulp above 1: tie, to even
    (1.0, 3 * 2.0 ** -8, 1.015625),             # tie between 1+2^-7 and 1+2^-6: to even
    (1.0, 2.0 ** -8 + 2.0 ** -40, 1.0078125),   # just above the tie: up (one rounding of
                                                # the exact sum, not of a rounded block)
    (-1.0, -(2.0 ** -8), -1.0),
    (0.5, -0.5, 0.0),
])
def test_residual_add_rounds_the_exact_sum_once(resid, block, want):
    H = 4
    r_out, _ = oracle.add_rmsnorm(np.tile(bf16([resid] * H), (1, 1)),
                                  np.full((1, H), block), bf16([1.0] * H), 1e-6)
    assert (f(r_out) == want).all()


def test_tokens_are_independent():
    H = 256
    g = gamma(H, seed=11)
    resid = W.bf16_normal((5, H), W.stream_key(12, "misc"), 1.0)
    block = W.normal(5 * H, W.stream_key(13, "misc")).reshape(5, H)
    r_all, x_all = oracle.add_rmsnorm(resid, block, g, 1e-6)
    for t in range(5):
        r_t, x_t = oracle.add_rmsnorm(resid[t:t + 1], block[t:t + 1], g, 1e-6)
        assert np.array_equal(r_t[0], r_all[t]) and np.array_equal(x_t[0], x_all[t])
