"""GPU parity of the fp32 tensor-core path (headdim 64, d_state 64, chunk
128; every product as three bf16 tcgen05 MMAs over hi/lo splits) against the
float64 oracle at the fp32 tolerance, on every output; the kernels that ran
are checked through the trace.
"""
import numpy as np
import pytest

from state_space_model_analytic_gb300 import synth

from parity_util import TOL, compare, rel_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

TC32_FWD = {"chunk_state_tc32", "state_pass_fwd", "chunk_scan_tc32"}
TC32_BWD = {"chunk_dstate_tc32", "state_pass_bwd", "bwd_x_tc32", "bwd_bc_tc32", "sum_bc_tc32",
            "reduce_heads"}


@pytest.fixture(scope="module")
def nat():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import _native
    from state_space_model_analytic_gb300 import build
    build()
    return _native


def traced_run(nat, dims, dev, history="given"):
    nat.trace_begin(64)
    try:
        out = run_gpu(dims, dev, history)
    finally:
        nat.trace_end()
    names = {r["name"] for r in nat.trace_read()}
    nat.trace_reset()
    return out, names


CASES = [
    # (B, T, H, G, h0, dt mode)
    (1, 128, 2, 1, False, "softplus"),      # one chunk
    (2, 512, 3, 1, True, "softplus"),       # odd head count
    (1, 384, 4, 2, True, "decay_span"),     # decays down to 1e-4 per step
    (2, 256, 6, 3, True, "softplus"),       # three groups
    (1, 1024, 24, 1, False, "softplus"),    # several head segments of the dB, dC kernel
    (1, 256, 8, 8, True, "softplus"),       # one head per group
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}t{}h{}g{}{}{}".format(
    c[0], c[1], c[2], c[3], "_h0" if c[4] else "", "_" + c[5]))
def test_tc32_every_output_against_oracle(nat, case):
    Bz, T, H, G, h0, mode = case
    dims = synth.Dims(Bz, T, H, 64, 64, G, 128, "f32")
    assert nat.lib().ssd_kernel_path(nat.make_dims(Bz, T, H, 64, 64, G, 128, False)) == 1
    inp = synth.make_inputs(dims, 100 + T + H, h0, mode)
    gpu, names = traced_run(nat, dims, to_device(dims, inp))
    assert TC32_FWD | TC32_BWD <= names, names
    ref = run_oracle(dims, inp)
    errs, bad = compare(gpu, ref, TOL["f32"])
    print(case, {k: f"{v:.1e}" for k, v in errs.items()})
    assert not bad, errs
    nat.check(nat.lib().ssd_device_status())


def test_tc32_recompute_mode_bitwise_and_repeatable(nat):
    dims = synth.Dims(2, 512, 4, 64, 64, 2, 128, "f32")
    inp = synth.make_inputs(dims, 31, True, "softplus")
    dev = to_device(dims, inp)
    a, names = traced_run(nat, dims, dev, "given")
    b, names_r = traced_run(nat, dims, dev, "recompute")
    assert "chunk_state_tc32" in names_r
    c = run_gpu(dims, dev, "given")
    for k in a:
        assert np.array_equal(a[k], b[k]), k
        assert np.array_equal(a[k], c[k]), k


def test_tc32_agrees_with_simt_path(nat):
    dims = synth.Dims(1, 512, 4, 64, 64, 1, 128, "f32")
    inp = synth.make_inputs(dims, 37, True, "softplus")
    dev = to_device(dims, inp)
    tc = run_gpu(dims, dev)
    nat.check(nat.lib().ssd_force_kernel_path(0))
    try:
        simt, names = traced_run(nat, dims, dev)
    finally:
        nat.check(nat.lib().ssd_force_kernel_path(-1))
    assert not any(n.endswith("_tc32") for n in names), names
    for k in tc:
        assert rel_err(tc[k], simt[k]) < TOL["f32"], k
