"""Pins of the oracle's dt / A preprocessing (dt = softplus(dt_raw + dt_bias),
A = -exp(a_log)) and of its chain rule back to dt_raw, dt_bias and a_log,
as in ``tensorized_mamba2_backward_impl`` and ``ssd_backward_reference``
(burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs)."""
import math

import numpy as np
import pytest

from oracle import dtprep


def rand_raw(seed, Bz, T, H, P, N, G):
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.standard_normal((Bz, T, H, P)),
        dt_raw=rng.uniform(-6.0, 3.0, size=(Bz, T, H)),  # softplus from ~0.0025 to ~3
        dt_bias=rng.uniform(-1.0, 0.5, size=H),
        a_log=rng.uniform(-0.7, 1.1, size=H),
        B=rng.standard_normal((Bz, T, G, N)) / np.sqrt(N),
        C=rng.standard_normal((Bz, T, G, N)) / np.sqrt(N),
        D=rng.uniform(0.5, 1.5, size=H),
        h0=rng.standard_normal((Bz, H, P, N)) * 0.3,
        dy=rng.standard_normal((Bz, T, H, P)),
    )


def loss(p):
    y, _, _ = dtprep.ssd_forward_raw(p["x"], p["dt_raw"], p["dt_bias"], p["a_log"], p["B"], p["C"],
                                     p["D"], p["h0"], chunk=4)
    return float(np.sum(p["dy"] * y))


@pytest.mark.parametrize("shape", [(1, 6, 2, 2, 3, 1), (2, 5, 4, 2, 2, 2)])
def test_raw_gradients_central_differences_every_element(shape):
    p = rand_raw(11, *shape)
    g = dtprep.ssd_backward_raw(p["x"], p["dt_raw"], p["dt_bias"], p["a_log"], p["B"], p["C"],
                                p["D"], p["h0"], p["dy"])
    for k, gk in (("dt_raw", "d_dt_raw"), ("dt_bias", "d_dt_bias"), ("a_log", "d_a_log")):
        base = p[k]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            q = dict(p)
            q[k] = base.copy(); q[k][idx] += eps
            lp = loss(q)
            q[k] = base.copy(); q[k][idx] -= eps
            lm = loss(q)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(g[gk] - fd)) / np.max(np.abs(fd))
        assert err < 1e-7, (k, err)


def test_raw_forward_T1_hand_case():
    """One step, one head: y = dt (C.B) x + exp(dt A) (h0 C) + D x with
    dt = log(1 + e^(dt_raw + dt_bias)) and A = -e^a_log, in scalar math."""
    rng = np.random.default_rng(5)
    P, N = 3, 4
    x = rng.standard_normal((1, 1, 1, P))
    Bm = rng.standard_normal((1, 1, 1, N))
    Cm = rng.standard_normal((1, 1, 1, N))
    h0 = rng.standard_normal((1, 1, P, N))
    D = np.array([0.7])
    dt_raw, dt_bias, a_log = np.array([[[0.4]]]), np.array([-1.3]), np.array([0.25])
    y, _, _ = dtprep.ssd_forward_raw(x, dt_raw, dt_bias, a_log, Bm, Cm, D, h0, chunk=1)
    dt = math.log1p(math.exp(0.4 - 1.3))
    A = -math.exp(0.25)
    cb = float(np.dot(Cm[0, 0, 0], Bm[0, 0, 0]))
    for p_ in range(P):
        want = dt * cb * x[0, 0, 0, p_] + math.exp(dt * A) * float(np.dot(h0[0, 0, p_], Cm[0, 0, 0])) \
            + 0.7 * x[0, 0, 0, p_]
        assert abs(y[0, 0, 0, p_] - want) < 1e-12


def test_softplus_and_sigmoid_extremes():
    z = np.array([-60.0, -5.0, 0.0, 5.0, 60.0])
    sp = dtprep.softplus(z)
    assert np.all(np.isfinite(sp))
    assert abs(sp[2] - math.log(2.0)) < 1e-15
    assert abs(sp[4] - 60.0) < 1e-12 and 0 < sp[0] < 1e-25
    for zi, si in zip(z[1:4], sp[1:4]):
        assert abs(si - math.log1p(math.exp(zi))) < 1e-14
    sg = dtprep.sigmoid(z)
    for zi, si in zip(z, sg):
        assert abs(si - 1.0 / (1.0 + math.exp(-zi))) < 1e-15
