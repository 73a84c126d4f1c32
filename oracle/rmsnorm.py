"""Gated RMSNorm after the SSD core, float64 (TEST INFRASTRUCTURE ONLY: used
by the tests and the benchmark's CPU baseline, never by the CUDA library).

Burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs:
``tensorized_mamba2_backward_impl`` forms inv_rms = 1 / sqrt(mean(y^2) + eps)
over each row; ``rmsnorm_gated_forward_from_inv_rms`` gives
out = (y * inv_rms) * weight * silu(z), and
``rmsnorm_gated_backward_from_inv_rms`` its gradients w.r.t. y, z and
weight, written out here in the page's order of steps.
"""
from __future__ import annotations

import numpy as np


def _sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def inv_rms(y, eps):
    y = np.asarray(y, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(y * y, axis=-1) + eps)


def forward(y, z, weight, eps):
    """Returns (out, inv_rms); rows are every index but the last."""
    y = np.asarray(y, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    inv = inv_rms(y, eps)
    out = (y * inv[..., None]) * w * (z * _sigmoid(z))
    return out, inv


def backward(y, z, weight, eps, dout):
    """dict dy, dz, dweight for the gradient dout of out."""
    y = np.asarray(y, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    g = np.asarray(dout, dtype=np.float64)
    width = y.shape[-1]
    inv = inv_rms(y, eps)[..., None]
    normalized = y * inv
    s = _sigmoid(z)
    gate = z * s
    weighted = normalized * w
    grad_weighted = g * gate
    grad_gate = g * weighted
    dweight = (grad_weighted * normalized).reshape(-1, width).sum(axis=0)
    grad_normalized = grad_weighted * w
    dot = np.sum(grad_normalized * y, axis=-1, keepdims=True)
    dy = grad_normalized * inv - y * dot * inv ** 3 / width
    dz = grad_gate * (s * (1.0 + z * (1.0 - s)))
    return {"dy": dy, "dz": dz, "dweight": dweight}
