"""GPU parity of the causal depthwise conv1d + SiLU (the step before the SSD
core) against the float64 oracle, through the C ABI."""
import numpy as np
import pytest

from oracle import conv
from state_space_model_analytic_gb300 import synth

from parity_util import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import build
    build()


def run_gpu(inp, dtype):
    import torch
    import state_space_model_analytic_gb300 as ssd
    io = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = lambda a, dt_: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dt_)
    x, g = t(inp["x"], io), t(inp["dout"], io)
    w, b, init = t(inp["weight"], torch.float32), t(inp["bias"], torch.float32), \
        t(inp["init_state"], torch.float32)
    out = ssd.conv1d_silu_forward(x, w, b, init)
    grads = ssd.conv1d_silu_backward(x, w, b, init, g)
    torch.cuda.synchronize()
    res = {"out": out, **grads}
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in res.items()}


def run_ref(inp):
    out = conv.forward(inp["x"], inp["weight"], inp["bias"], inp["init_state"])
    return {"out": out, **conv.backward(inp["x"], inp["weight"], inp["bias"], inp["init_state"],
                                        inp["dout"])}


CASES = [  # (B, T, C, K, dtype, init): every K, ragged tiles along time (T not a
    # multiple of the tile), several CTAs along time and channels with a partial last one
    (1, 5, 8, 4, "f32", True), (2, 130, 12, 4, "f32", False), (3, 64, 16, 3, "bf16", True),
    (1, 200, 40, 2, "bf16", True), (2, 97, 24, 1, "f32", True), (2, 333, 264, 4, "bf16", True),
    (1, 700, 136, 3, "f32", False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) + c[4])
def test_conv1d_silu_every_output(case):
    Bz, T, C, K, dtype, init = case
    inp = synth.conv_inputs(Bz, T, C, K, dtype, 3 + T + C, init)
    gpu = run_gpu(inp, dtype)
    ref = run_ref(inp)
    errs = {k: rel_err(gpu[k], ref[k]) for k in ref}
    assert all(v <= TOL[dtype] for v in errs.values()), errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv1d_silu_without_bias(dtype):
    """bias NULL: the pre-activation has no bias term; dbias is still the sum
    of the gradients of the pre-activation."""
    inp = synth.conv_inputs(2, 300, 136, 3, dtype, 77, True)
    inp["bias"] = None
    gpu = run_gpu(inp, dtype)
    ref = run_ref(inp)
    errs = {k: rel_err(gpu[k], ref[k]) for k in ref}
    assert all(v <= TOL[dtype] for v in errs.values()), errs


def test_conv1d_silu_full_size_xbc_deterministic():
    """xBC of the bf16 d_inner-2048 workload: B = 4, T = 2048, C = H*P +
    2*G*N = 2304, d_conv = 4; every output against the oracle, and two runs
    equal bit for bit."""
    inp = synth.conv_inputs(4, 2048, 2304, 4, "bf16", 2304)
    a = run_gpu(inp, "bf16")
    b = run_gpu(inp, "bf16")
    ref = run_ref(inp)
    errs = {k: rel_err(a[k], ref[k]) for k in ref}
    print("conv1d full size: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_conv1d_rejects_unsupported():
    import torch
    import state_space_model_analytic_gb300 as ssd
    from state_space_model_analytic_gb300 import _native as nat
    x = torch.zeros(1, 8, 12, dtype=torch.bfloat16, device="cuda")  # 12 not a multiple of 8
    with pytest.raises(nat.SsdError):
        ssd.conv1d_silu_forward(x, torch.zeros(12, 4, device="cuda"))
    x = torch.zeros(1, 8, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nat.SsdError):  # d_conv 5
        ssd.conv1d_silu_forward(x, torch.zeros(16, 5, device="cuda"))
