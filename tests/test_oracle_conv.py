"""Pins of the conv1d + SiLU oracle (``depthwise_conv_preact_with_history``
and the fallback conv backward of ``tensorized_mamba2_backward_impl``,
burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs): central
differences, the one-tap and shifted-tap special cases in scalar math, and
splitting the sequence with the initial state carrying the history."""
import math

import numpy as np
import pytest

from oracle import conv


def rand(seed, Bz, T, C, K, init=True):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Bz, T, C)), rng.standard_normal((C, K)) * 0.7,
            rng.standard_normal(C) * 0.3,
            rng.standard_normal((Bz, C, K)) if init else None, rng.standard_normal((Bz, T, C)))


@pytest.mark.parametrize("K", [1, 3, 4])
def test_gradients_central_differences_every_element(K):
    x, w, b, init, g = rand(K, 2, 7, 3, K)

    def loss(x_, w_, b_):
        return float(np.sum(g * conv.forward(x_, w_, b_, init)))

    grads = conv.backward(x, w, b, init, g)
    for name, base, key in (("x", x, "dx"), ("w", w, "dweight"), ("b", b, "dbias")):
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            h = 1e-6 * max(1.0, abs(base[idx]))
            args = {"x": x, "w": w, "b": b}
            plus = base.copy(); plus[idx] += h
            minus = base.copy(); minus[idx] -= h
            args[name] = plus
            lp = loss(args["x"], args["w"], args["b"])
            args[name] = minus
            lm = loss(args["x"], args["w"], args["b"])
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(grads[key] - fd)) / np.max(np.abs(fd))
        assert err < 1e-7, (name, err)


def test_one_tap_is_pointwise_silu():
    x, _, _, _, _ = rand(5, 1, 6, 2, 1, init=False)
    w = np.array([[2.0], [-0.5]])
    b = np.array([0.1, 0.0])
    out = conv.forward(x, w, b)
    for t in range(6):
        for c in range(2):
            p = w[c, 0] * x[0, t, c] + b[c]
            assert abs(out[0, t, c] - p / (1.0 + math.exp(-p))) < 1e-14


def test_first_tap_reaches_back_k_minus_1_steps_into_the_state():
    """Weight only on tap 0: the output at step t reads the input K - 1 steps
    back, and the last K - 1 entries of the initial state before step K - 1."""
    K, T = 4, 9
    x, _, _, init, _ = rand(6, 1, T, 1, K)
    w = np.zeros((1, K)); w[0, 0] = 1.0
    out = conv.forward(x, w, None, init)
    for t in range(T):
        src = x[0, t - (K - 1), 0] if t >= K - 1 else init[0, 0, t + 1]
        assert abs(out[0, t, 0] - src / (1.0 + math.exp(-src))) < 1e-14


def test_split_sequence_with_carried_state():
    """conv(x) over T steps equals conv of the second part started from the
    last K inputs of the first part (the history the page concatenates)."""
    K = 4
    x, w, b, _, _ = rand(7, 2, 12, 3, K, init=False)
    full = conv.forward(x, w, b)
    T1 = 5
    carry = np.transpose(x[:, T1 - K:T1, :], (0, 2, 1))  # [B, C, K]
    second = conv.forward(x[:, T1:, :], w, b, carry)
    np.testing.assert_allclose(second, full[:, T1:, :], rtol=1e-14, atol=1e-14)
