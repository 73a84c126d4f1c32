"""Pins of the gated-RMSNorm oracle (``rmsnorm_gated_forward_from_inv_rms`` /
``rmsnorm_gated_backward_from_inv_rms``, burn_dragon_kernel 0.5.0,
src/sequence/mamba2/backward.rs) to facts that do not come from it:
central differences, scale invariance in y, the unit mean square of the
normalized rows, and a scalar hand case."""
import math

import numpy as np
import pytest

from oracle import rmsnorm


def rand(seed, rows, width):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, width)) * 1.7, rng.standard_normal((rows, width)) * 2.0,
            rng.uniform(0.5, 1.5, size=width), rng.standard_normal((rows, width)))


@pytest.mark.parametrize("eps", [1e-5, 0.3])
def test_gradients_central_differences_every_element(eps):
    y, z, w, g = rand(1, 3, 8)

    def loss(y_, z_, w_):
        out, _ = rmsnorm.forward(y_, z_, w_, eps)
        return float(np.sum(g * out))

    grads = rmsnorm.backward(y, z, w, eps, g)
    for name, base, key in (("y", y, "dy"), ("z", z, "dz"), ("w", w, "dweight")):
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            h = 1e-6 * max(1.0, abs(base[idx]))
            args = {"y": y, "z": z, "w": w}
            plus = base.copy(); plus[idx] += h
            minus = base.copy(); minus[idx] -= h
            args[name] = plus
            lp = loss(args["y"], args["z"], args["w"])
            args[name] = minus
            lm = loss(args["y"], args["z"], args["w"])
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(grads[key] - fd)) / np.max(np.abs(fd))
        assert err < 1e-7, (name, err)


def test_scale_invariance_and_unit_mean_square():
    """With eps = 0 the output does not change when a row of y is scaled, so
    sum_w y dy = 0 per row; the normalized rows have mean square 1."""
    y, z, w, g = rand(2, 4, 16)
    out1, inv1 = rmsnorm.forward(y, z, w, 0.0)
    out2, _ = rmsnorm.forward(y * 3.5, z, w, 0.0)
    np.testing.assert_allclose(out1, out2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(np.mean((y * inv1[:, None]) ** 2, axis=-1), 1.0, rtol=1e-14)
    d = rmsnorm.backward(y, z, w, 0.0, g)
    assert np.max(np.abs(np.sum(y * d["dy"], axis=-1))) < 1e-12


def test_hand_case_width_two():
    y = np.array([[3.0, 4.0]])
    z = np.array([[0.0, 1.0]])
    w = np.array([2.0, 0.5])
    out, inv = rmsnorm.forward(y, z, w, 0.0)
    r = math.sqrt((9.0 + 16.0) / 2.0)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(inv[0] - 1.0 / r) < 1e-15
    assert out[0, 0] == 0.0  # silu(0) = 0
    assert abs(out[0, 1] - 4.0 / r * 0.5 * silu1) < 1e-15
