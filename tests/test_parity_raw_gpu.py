"""GPU parity of the raw-dt entry points (dt = softplus(dt_raw + dt_bias),
A = -exp(a_log) on the device; gradients w.r.t. dt_raw, dt_bias, a_log)
against the float64 oracle's preprocessing composed with the oracle core."""
import numpy as np
import pytest

from oracle import dtprep
from state_space_model_analytic_gb300 import synth

from parity_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import build
    build()


def run_raw(dims, inp, history="given"):
    import torch
    import state_space_model_analytic_gb300 as ssd
    dev = to_device(dims, inp)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    raw = {k: f32(inp[k]) for k in ("dt_raw", "dt_bias", "a_log")}
    y, fs, cs = ssd.forward_raw(dev["x"], raw["dt_raw"], raw["dt_bias"], raw["a_log"], dev["B"],
                                dev["C"], dev["D"], dev["h0"], chunk=dims.chunk)
    g = ssd.backward_raw(dev["x"], raw["dt_raw"], raw["dt_bias"], raw["a_log"], dev["B"],
                         dev["C"], dev["D"], dev["h0"], dev["dy"],
                         cs if history == "given" else None, chunk=dims.chunk)
    torch.cuda.synchronize()
    out = {"y": y, "final_state": fs, "chunk_states": cs, **g}
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in out.items() if v is not None}


def run_oracle_raw(dims, inp):
    y, fs, cs = dtprep.ssd_forward_raw(inp["x"], inp["dt_raw"], inp["dt_bias"], inp["a_log"],
                                       inp["B"], inp["C"], inp["D"], inp["h0"], chunk=dims.chunk)
    g = dtprep.ssd_backward_raw(inp["x"], inp["dt_raw"], inp["dt_bias"], inp["a_log"], inp["B"],
                                inp["C"], inp["D"], inp["h0"], inp["dy"])
    return {"y": y, "final_state": fs, "chunk_states": cs, **g}


KEYS = ("y", "final_state", "chunk_states", "dx", "d_dt_raw", "d_dt_bias", "d_a_log", "dB", "dC",
        "dD", "dh0")

CASES = [
    (1, 128, 3, 16, 48, 3, 64, "f32", True),
    (2, 256, 4, 32, 32, 2, 32, "f32", False),
    (1, 512, 4, 64, 128, 2, 256, "bf16", True),
    (2, 256, 6, 64, 128, 3, 128, "bf16", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:7])) + c[7])
@pytest.mark.parametrize("history", ["given", "recompute"])
def test_raw_entry_points_every_output(case, history):
    Bz, T, H, P, N, G, Q, dt_, h0 = case
    dims = synth.Dims(Bz, T, H, P, N, G, Q, dt_)
    inp = synth.make_inputs(dims, 31 + T + H, h0, "softplus")
    gpu = run_raw(dims, inp, history)
    ref = run_oracle_raw(dims, inp)
    errs = {k: rel_err(gpu[k], ref[k]) for k in KEYS}
    bad = {k: v for k, v in errs.items() if not v <= TOL[dt_]}
    assert not bad, errs


@pytest.mark.parametrize("q,h0,history", [(128, True, "recompute"), (256, True, "given"),
                                           (128, False, "given"), (256, False, "recompute")])
def test_raw_entry_points_fused_path(q, h0, history):
    """Shapes with enough (b, h) pairs for the fused tensor-core path, where the
    raw-dt transforms run inside the step's kernels (the forward, the state
    scans, the backward): it must be those kernels that ran; every output
    against the oracle, with an initial state or without, history given or
    recomputed, several chunks and groups."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(4, 512, 64, 64, 128, 16, q, "bf16")  # B * H = 256 (b, h) pairs
    inp = synth.make_inputs(dims, 41 + q, h0, "softplus")
    nat.trace_begin(64)
    try:
        gpu = run_raw(dims, inp, history)
    finally:
        nat.trace_end()
    names = [r["name"] for r in nat.trace_read()]
    nat.trace_reset()
    assert "fwd_single_tc" in names and "bwd_tc" in names and "dt_prep" not in names, names
    ref = run_oracle_raw(dims, inp)
    errs = {k: rel_err(gpu[k], ref[k]) for k in KEYS if k in gpu}
    bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
    assert not bad, errs
    nat.check(nat.lib().ssd_device_status())


def test_raw_entry_points_full_size_bf16_d_inner_2048():
    """The benchmark workload (B4 T2048 H32 P64 N128 G1 Q256) through the
    raw entry points, every output against the oracle."""
    dims, inp = synth.config_inputs(1)
    gpu = run_raw(dims, inp)
    ref = run_oracle_raw(dims, inp)
    errs = {k: rel_err(gpu[k], ref[k]) for k in KEYS if k in gpu}
    print("raw config 1: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
