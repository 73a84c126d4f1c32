"""Causal depthwise conv1d + SiLU on xBC, float64 (TEST INFRASTRUCTURE ONLY:
used by the tests and the benchmark's CPU baseline, never by the CUDA
library).

Burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs:
``depthwise_conv_preact_with_history`` concatenates the initial conv state
(d_conv entries per channel, zeros when absent) in front of the input and
sums, per tap, the window starting one step after the tap index times the
tap's weight, plus the bias; the output is silu of that.  The fallback conv
backward of ``tensorized_mamba2_backward_impl`` multiplies the output
gradient by silu', sums it for the bias, sums its products with the windows
for each tap's weight, and scatters it through the weights back onto the
history, whose input part is the gradient w.r.t. x.

Layouts as in the library: x, dout [B,T,C]; weight [C,K]; bias [C];
init_state [B,C,K].
"""
from __future__ import annotations

import numpy as np


def _sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def _history(x, init_state, K):
    """[B, C, K + T]: the initial state, then x over time."""
    x = np.asarray(x, dtype=np.float64)
    Bz, T, C = x.shape
    init = np.zeros((Bz, C, K)) if init_state is None else np.asarray(init_state, dtype=np.float64)
    return np.concatenate([init, np.transpose(x, (0, 2, 1))], axis=2)


def preact(x, weight, bias, init_state):
    w = np.asarray(weight, dtype=np.float64)
    C, K = w.shape
    h = _history(x, init_state, K)
    T = h.shape[2] - K
    p = np.zeros((h.shape[0], C, T))
    for tap in range(K):
        p += h[:, :, tap + 1:tap + 1 + T] * w[None, :, tap, None]
    if bias is not None:
        p += np.asarray(bias, dtype=np.float64)[None, :, None]
    return p, h  # [B, C, T], [B, C, K + T]


def forward(x, weight, bias=None, init_state=None):
    p, _ = preact(x, weight, bias, init_state)
    return np.transpose(p * _sigmoid(p), (0, 2, 1))


def backward(x, weight, bias, init_state, dout):
    """dict dx [B,T,C], dweight [C,K], dbias [C]."""
    w = np.asarray(weight, dtype=np.float64)
    C, K = w.shape
    p, h = preact(x, weight, bias, init_state)
    T = p.shape[2]
    s = _sigmoid(p)
    gp = np.transpose(np.asarray(dout, dtype=np.float64), (0, 2, 1)) * (s * (1.0 + p * (1.0 - s)))
    dbias = gp.sum(axis=(0, 2))
    dweight = np.zeros((C, K))
    gh = np.zeros_like(h)
    for tap in range(K):
        dweight[:, tap] = (gp * h[:, :, tap + 1:tap + 1 + T]).sum(axis=(0, 2))
        gh[:, :, tap + 1:tap + 1 + T] += gp * w[None, :, tap, None]
    dx = np.transpose(gh[:, :, K:K + T], (0, 2, 1))
    return {"dx": dx, "dweight": dweight, "dbias": dbias}
