"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test targets a different plausible mistake: a dropped term or wrong
sign in the backward (finite differences, autograd of an independent
recurrence, homogeneity identities), a wrong decay index or an off-by-one
in the history (the quadratic form, the history semantics), and wrong
bookkeeping of the sums over heads, batch and time (closed forms).
The recurrence being pinned is the one of ``ssd_forward_state_history_reference``
and ``ssd_backward_reference`` (burn_dragon_kernel 0.5.0,
src/sequence/mamba2/backward.rs).
"""
import numpy as np
import pytest

from oracle import dual
from state_space_model_analytic_gb300 import synth


def rand_problem(seed, Bz, T, H, P, N, G, h0=True, a_scale=1.0):
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.standard_normal((Bz, T, H, P)),
        dt=rng.uniform(0.05, 0.8, size=(Bz, T, H)),
        A=-rng.uniform(0.5, 3.0, size=H) * a_scale,
        B=rng.standard_normal((Bz, T, G, N)) / np.sqrt(N),
        C=rng.standard_normal((Bz, T, G, N)) / np.sqrt(N),
        D=rng.uniform(0.5, 1.5, size=H),
        h0=(rng.standard_normal((Bz, H, P, N)) * 0.3) if h0 else None,
        dy=rng.standard_normal((Bz, T, H, P)),
    )


def fwd(o, p, chunk=4):
    return o.ssd_forward(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["h0"], chunk=chunk)


def bwd(o, p):
    return o.ssd_backward(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["h0"], p["dy"])


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --- forward ---------------------------------------------------------------

@pytest.mark.parametrize("h0", [False, True])
def test_forward_matches_quadratic_form(oracle_mod, h0):
    p = rand_problem(1, 2, 12, 4, 3, 5, 2, h0=h0)
    y, fs, cs = fwd(oracle_mod, p, chunk=4)
    y_ref, st_ref = dual.forward(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["h0"])
    assert rel(y, y_ref) < 1e-12
    assert rel(fs, st_ref[:, -1]) < 1e-12
    # history entry c is the state before step c*Q: h0 (or zeros), then states after step c*Q-1
    start = p["h0"] if h0 else np.zeros_like(fs)
    assert np.array_equal(cs[:, 0], start)
    for c in range(1, 3):
        assert rel(cs[:, c], st_ref[:, c * 4 - 1]) < 1e-12


def test_T1_hand_case(oracle_mod):
    p = rand_problem(2, 1, 1, 1, 3, 4, 1, h0=True)
    y, fs, _ = fwd(oracle_mod, p, chunk=1)
    x, dt, A, B, C, D, h0, dy = (p[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy"))
    e = np.exp(dt[0, 0, 0] * A[0])
    cb = float(C[0, 0, 0] @ B[0, 0, 0])
    xv, dyv, h0m = x[0, 0, 0], dy[0, 0, 0], h0[0, 0]
    y_hand = dt[0, 0, 0] * cb * xv + e * (h0m @ C[0, 0, 0]) + D[0] * xv
    assert rel(y[0, 0, 0], y_hand) < 1e-13
    g = bwd(oracle_mod, p)
    gS = np.outer(dyv, C[0, 0, 0])
    h1 = e * h0m + dt[0, 0, 0] * np.outer(xv, B[0, 0, 0])
    assert rel(g["dx"][0, 0, 0], D[0] * dyv + dt[0, 0, 0] * cb * dyv) < 1e-13
    assert rel(g["ddt"][0, 0, 0], cb * (xv @ dyv) + np.sum(gS * h0m) * e * A[0]) < 1e-13
    assert rel(g["dA"][0], np.sum(gS * h0m) * e * dt[0, 0, 0]) < 1e-13
    assert rel(g["dB"][0, 0, 0], dt[0, 0, 0] * (xv @ dyv) * C[0, 0, 0]) < 1e-13
    assert rel(g["dC"][0, 0, 0], h1.T @ dyv) < 1e-13
    assert rel(g["dh0"][0, 0], e * gS) < 1e-13
    assert rel(g["dD"][0], xv @ dyv) < 1e-13


# --- backward --------------------------------------------------------------

def loss(o, p):
    y, _, _ = fwd(o, p)
    return float(np.sum(p["dy"] * y))


@pytest.mark.parametrize("shape", [(1, 8, 2, 2, 3, 1), (1, 7, 4, 2, 3, 2)])
def test_backward_central_differences_every_element(oracle_mod, shape):
    p = rand_problem(3, *shape, h0=True)
    g = bwd(oracle_mod, p)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "h0": "dh0"}
    for k, gk in names.items():
        base = p[k]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            q = dict(p)
            q[k] = base.copy(); q[k][idx] += eps
            lp = loss(oracle_mod, q)
            q[k] = base.copy(); q[k][idx] -= eps
            lm = loss(oracle_mod, q)
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel(g[gk], fd) < 1e-7, k


def torch_recurrence_grads(p):
    """Gradients by torch autograd of a plain float64 step loop written here
    (an independent route from the hand-derived reverse sweep)."""
    import torch
    t = {k: (None if v is None else torch.tensor(v, dtype=torch.float64, requires_grad=True))
         for k, v in p.items() if k != "dy"}
    x, dt, A, B, C, D, h0 = (t[k] for k in ("x", "dt", "A", "B", "C", "D", "h0"))
    Bz, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    Bh = B.repeat_interleave(hpg, dim=2)  # [B,T,H,N]
    Ch = C.repeat_interleave(hpg, dim=2)
    s = h0 if h0 is not None else torch.zeros(Bz, H, P, N, dtype=torch.float64)
    ys = []
    for step in range(T):
        dec = torch.exp(dt[:, step] * A)[:, :, None, None]
        s = s * dec + (dt[:, step, :, None, None] * x[:, step, :, :, None] * Bh[:, step, :, None, :])
        ys.append((s * Ch[:, step, :, None, :]).sum(-1) + D[None, :, None] * x[:, step])
    y = torch.stack(ys, 1)
    (y * torch.tensor(p["dy"])).sum().backward()
    out = {"d" + k: t[k].grad.numpy() for k in ("x", "dt", "A", "B", "C", "D")}
    out["dh0"] = t["h0"].grad.numpy() if h0 is not None else None
    return y.detach().numpy(), out


@pytest.mark.parametrize("h0", [True, False])
def test_backward_matches_autograd_of_recurrence(oracle_mod, h0):
    p = rand_problem(4, 2, 40, 4, 4, 6, 2, h0=h0)
    y_t, gt = torch_recurrence_grads(p)
    y, _, _ = fwd(oracle_mod, p)
    assert rel(y, y_t) < 1e-12
    g = bwd(oracle_mod, p)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        assert rel(g[k], gt[k]) < 1e-11, k
    if h0:
        assert rel(g["dh0"], gt["dh0"]) < 1e-11


def test_A_zero_closed_form(oracle_mod):
    """With A = 0 every decay is 1: the state is a running sum of
    dt_s x_s B_s^T and every gradient is a (reverse) cumulative sum."""
    p = rand_problem(5, 2, 9, 4, 3, 5, 2, h0=True)
    p["A"] = np.zeros(4)
    x, dt, B, C, D, h0, dy = (p[k] for k in ("x", "dt", "B", "C", "D", "h0", "dy"))
    hpg = 2
    Bh = np.repeat(B, hpg, axis=2)
    Ch = np.repeat(C, hpg, axis=2)
    drive = dt[..., None, None] * x[..., :, None] * Bh[..., None, :]      # [B,T,H,P,N]
    states = h0[:, None] + np.cumsum(drive, axis=1)
    prev = np.concatenate([h0[:, None], states[:, :-1]], axis=1)
    y_cf = np.einsum("bthpn,bthn->bthp", states, Ch) + D[None, None, :, None] * x
    y, fs, _ = fwd(oracle_mod, p)
    assert rel(y, y_cf) < 1e-12 and rel(fs, states[:, -1]) < 1e-12
    outer = dy[..., :, None] * Ch[..., None, :]                           # dy_t C_t^T
    Gs = np.flip(np.cumsum(np.flip(outer, 1), axis=1), 1)                 # sum_{t>=s}
    g = bwd(oracle_mod, p)
    GB = np.einsum("bthpn,bthn->bthp", Gs, Bh)
    assert rel(g["dx"], D[None, None, :, None] * dy + dt[..., None] * GB) < 1e-12
    assert rel(g["ddt"], np.einsum("bthp,bthp->bth", x, GB)) < 1e-12
    assert rel(g["dA"], np.einsum("bth,bthpn->h", dt, Gs * prev)) < 1e-12
    dBh = dt[..., None] * np.einsum("bthpn,bthp->bthn", Gs, x)
    dCh = np.einsum("bthpn,bthp->bthn", states, dy)
    Bsz, T, G, N = B.shape
    assert rel(g["dB"], dBh.reshape(Bsz, T, G, hpg, N).sum(3)) < 1e-12
    assert rel(g["dC"], dCh.reshape(Bsz, T, G, hpg, N).sum(3)) < 1e-12
    assert rel(g["dh0"], Gs[:, 0]) < 1e-12
    assert rel(g["dD"], np.einsum("bthp,bthp->h", dy, x)) < 1e-12


def test_homogeneity_identities(oracle_mod):
    """(i) degree-1 homogeneity in (x, h0); (ii) invariance under
    dt->l*dt, A->A/l, x->x/l, D->l*D per head; (iii) invariance under
    B->m*B, C->C/m, h0->m*h0 per group."""
    p = rand_problem(6, 2, 33, 6, 4, 5, 3, h0=True)
    y, _, _ = fwd(oracle_mod, p)
    g = bwd(oracle_mod, p)
    L = np.sum(p["dy"] * y)
    lhs = np.sum(p["x"] * g["dx"]) + np.sum(p["h0"] * g["dh0"])
    assert abs(lhs - L) < 1e-12 * max(1.0, abs(L)) * 100
    for h in range(6):
        v = (np.sum(p["dt"][..., h] * g["ddt"][..., h]) - p["A"][h] * g["dA"][h]
             - np.sum(p["x"][:, :, h] * g["dx"][:, :, h]) + p["D"][h] * g["dD"][h])
        assert abs(v) < 1e-10
    for gi in range(3):
        hs = range(gi * 2, gi * 2 + 2)
        v = (np.sum(p["B"][:, :, gi] * g["dB"][:, :, gi])
             + sum(np.sum(p["h0"][:, h] * g["dh0"][:, h]) for h in hs)
             - np.sum(p["C"][:, :, gi] * g["dC"][:, :, gi]))
        assert abs(v) < 1e-10


def test_dD_closed_form_and_linearity_in_dy(oracle_mod):
    p = rand_problem(7, 2, 10, 4, 3, 4, 2, h0=True)
    g1 = bwd(oracle_mod, p)
    assert rel(g1["dD"], np.einsum("bthp,bthp->h", p["dy"], p["x"])) < 1e-13
    q = dict(p); q["dy"] = 2.5 * p["dy"]
    g2 = bwd(oracle_mod, q)
    for k in g1:
        assert rel(g2[k], 2.5 * g1[k]) < 1e-13, k


def test_split_sequence_equivalence(oracle_mod):
    """ssd(x[0:T]) equals ssd(x[T1:T]) seeded with the final state of
    ssd(x[0:T1]); the second half's gradients match the full run's."""
    p = rand_problem(8, 2, 16, 4, 3, 5, 2, h0=True)
    T1 = 6
    first = {k: (v[:, :T1] if k in ("x", "dt", "B", "C", "dy") else v) for k, v in p.items()}
    y1, fs1, _ = fwd(oracle_mod, first)
    second = {k: (v[:, T1:] if k in ("x", "dt", "B", "C", "dy") else v) for k, v in p.items()}
    second["h0"] = fs1
    y2, fs2, _ = fwd(oracle_mod, second)
    y, fs, _ = fwd(oracle_mod, p)
    assert rel(np.concatenate([y1, y2], 1), y) < 1e-12 and rel(fs2, fs) < 1e-12
    gf = bwd(oracle_mod, p)
    g2 = bwd(oracle_mod, second)
    for k in ("dx", "ddt", "dB", "dC"):
        assert rel(g2[k], gf[k][:, T1:]) < 1e-12, k
    # the state gradient at the split, pushed back through the first half with
    # dy = 0 there, must reproduce the full run's dh0 contribution of the tail:
    # by linearity in dy, dh0_full = dh0(first, dy_first) + carry of g2's dh0.
    zero_tail = dict(p); zero_tail["dy"] = p["dy"].copy(); zero_tail["dy"][:, T1:] = 0
    g_head = bwd(oracle_mod, zero_tail)
    # pushing g2["dh0"] back through steps T1-1..0 multiplies by the decays
    decay = np.exp(np.cumsum(p["dt"][:, :T1] * p["A"], axis=1)[:, -1])  # [B,H]
    assert rel(gf["dh0"], g_head["dh0"] + decay[..., None, None] * g2["dh0"]) < 1e-12


def test_history_is_chunk_subsample(oracle_mod):
    p = rand_problem(9, 1, 24, 2, 3, 4, 1, h0=True)
    _, fs4, c4 = fwd(oracle_mod, p, chunk=4)
    _, fs8, c8 = fwd(oracle_mod, p, chunk=8)
    _, fs3, c3 = fwd(oracle_mod, p, chunk=3)
    assert np.array_equal(c4[:, ::2], c8) and np.array_equal(fs4, fs8)
    assert np.array_equal(c3[:, ::4], c4[:, ::3])


def test_thread_count_does_not_change_results(oracle_mod):
    p = rand_problem(10, 2, 20, 6, 3, 4, 2, h0=True)
    g1 = oracle_mod.ssd_backward(*(p[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")), threads=1)
    g5 = oracle_mod.ssd_backward(*(p[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")), threads=5)
    for k in g1:
        assert np.array_equal(g1[k], g5[k]), k


def test_long_decay_no_nan(oracle_mod):
    """Decays near 1e-4 over long spans underflow to zero without NaN."""
    d = synth.Dims(1, 600, 2, 4, 4, 1, 64, "f32")
    inp = synth.make_inputs(d, 11, True, "decay_span")
    y, fs, cs = oracle_mod.ssd_forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["h0"], chunk=64)
    g = oracle_mod.ssd_backward(*(inp[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")))
    assert np.isfinite(y).all() and np.isfinite(fs).all() and np.isfinite(cs).all()
    assert all(np.isfinite(v).all() for v in g.values())


def test_modular_case_golden(oracle_mod):
    """Regression pin against values the oracle wrote when it was pinned
    (tests/golden/make_golden.py; modular-pattern inputs of the Mamba-2
    backward page's parity tests)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "modular_case.json")
    rec = json.load(open(path))
    dims, inp = synth.modular_inputs(chunk=16)
    y, fs, cs = oracle_mod.ssd_forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["h0"], chunk=16)
    g = oracle_mod.ssd_backward(*(inp[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")))
    outs = {"y": y, "final_state": fs, "chunk_states": cs, **g}
    for k, s in rec["samples"].items():
        flat = outs[k].reshape(-1)
        assert list(outs[k].shape) == s["shape"]
        np.testing.assert_allclose(flat[s["index"]], s["value"], rtol=1e-12, atol=1e-12 * s["absmax"])
