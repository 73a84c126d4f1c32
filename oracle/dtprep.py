"""The dt and A preprocessing in front of the SSD core, float64
(TEST INFRASTRUCTURE ONLY: used by the tests, never by the CUDA library).

Burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs:
``tensorized_mamba2_backward_impl`` forms dt = softplus(dt_raw + dt_bias)
(the bias per head) and A = -exp(a_log), and in its backward multiplies the
gradient w.r.t. dt by sigmoid(dt_raw + dt_bias) (the derivative of
softplus) and sums that over batch and time for dt_bias;
``ssd_backward_reference`` returns the gradient w.r.t. a_log as the
gradient w.r.t. A summed over batch and time times -exp(a_log).
"""
from __future__ import annotations

import numpy as np

from .core import ssd_backward, ssd_forward


def softplus(z):
    """log(1 + e^z) without overflow."""
    return np.logaddexp(0.0, z)


def sigmoid(z):
    """1 / (1 + e^-z) without overflow (its tanh form)."""
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def preprocess(dt_raw, dt_bias, a_log):
    """dt [B,T,H] and A [H] of the core from the raw parameters."""
    dt_raw = np.asarray(dt_raw, dtype=np.float64)
    dt = softplus(dt_raw + np.asarray(dt_bias, dtype=np.float64)[None, None, :])
    A = -np.exp(np.asarray(a_log, dtype=np.float64))
    return dt, A


def ssd_forward_raw(x, dt_raw, dt_bias, a_log, B, C, D, h0=None, chunk=64, threads=None):
    dt, A = preprocess(dt_raw, dt_bias, a_log)
    return ssd_forward(x, dt, A, B, C, D, h0, chunk=chunk, threads=threads)


def ssd_backward_raw(x, dt_raw, dt_bias, a_log, B, C, D, h0, dy, threads=None):
    """dict dx, d_dt_raw, d_dt_bias, d_a_log, dB, dC, dD, dh0."""
    dt, A = preprocess(dt_raw, dt_bias, a_log)
    g = ssd_backward(x, dt, A, B, C, D, h0, dy, threads=threads)
    z = np.asarray(dt_raw, dtype=np.float64) + np.asarray(dt_bias, dtype=np.float64)[None, None, :]
    d_dt_raw = g["ddt"] * sigmoid(z)
    out = {k: v for k, v in g.items() if k not in ("ddt", "dA")}
    out["d_dt_raw"] = d_dt_raw
    out["d_dt_bias"] = d_dt_raw.sum(axis=(0, 1))
    out["d_a_log"] = g["dA"] * A
    return out
