"""Independent numpy restatement of the SSD forward as its quadratic form
(TEST INFRASTRUCTURE ONLY; brute force, tiny inputs).

Unrolling the recurrence of ``ssd_forward_state_history_reference``
(burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs) gives, with
a_r = dt_r * A_h and the group g of head h,

    y_t = sum_{s<=t} exp(sum_{s<r<=t} a_r) * (C_t . B_s) * dt_s * x_s
          + exp(sum_{r<=t} a_r) * (h0 C_t) + D_h * x_t,

    state after t = exp(sum_{r<=t} a_r) h0 + sum_{s<=t} exp(sum_{s<r<=t} a_r) dt_s x_s B_s^T.

This module evaluates those sums directly with O(T^2) loops over (t, s);
it shares nothing with the C oracle and is used only to pin it.
"""
from __future__ import annotations

import numpy as np


def _decay_sum(a, s, t):
    """sum_{s < r <= t} a_r, summed term by term."""
    return float(np.sum(a[s + 1:t + 1]))


def forward(x, dt, A, B, C, D, h0=None):
    Bz, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    y = np.zeros((Bz, T, H, P))
    states = np.zeros((Bz, T, H, P, N))  # state after each step
    for b in range(Bz):
        for h in range(H):
            g = h // hpg
            a = dt[b, :, h] * A[h]
            for t in range(T):
                st = np.zeros((P, N))
                if h0 is not None:
                    st += np.exp(_decay_sum(a, -1, t)) * h0[b, h]
                for s in range(t + 1):
                    w = np.exp(_decay_sum(a, s, t)) * dt[b, s, h]
                    st += w * np.outer(x[b, s, h], B[b, s, g])
                states[b, t, h] = st
                acc = np.zeros(P)
                if h0 is not None:
                    acc += np.exp(_decay_sum(a, -1, t)) * (h0[b, h] @ C[b, t, g])
                for s in range(t + 1):
                    w = np.exp(_decay_sum(a, s, t)) * dt[b, s, h]
                    acc += w * float(C[b, t, g] @ B[b, s, g]) * x[b, s, h]
                y[b, t, h] = acc + D[h] * x[b, t, h]
    return y, states
