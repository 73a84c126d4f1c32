"""GPU parity of the gated RMSNorm (the step after the SSD core) against the
float64 oracle, through the C ABI."""
import numpy as np
import pytest

from oracle import rmsnorm
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


def run_gpu(inp, dtype, eps, pass_inv=True):
    import torch
    import state_space_model_analytic_gb300 as ssd
    io = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = lambda a, dt_: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dt_)
    y, z, g = t(inp["y"], io), t(inp["z"], io), t(inp["dout"], io)
    w = t(inp["weight"], torch.float32)
    out, inv = ssd.rmsnorm_gated_forward(y, z, w, eps)
    grads = ssd.rmsnorm_gated_backward(y, z, w, eps, g, inv if pass_inv else None)
    torch.cuda.synchronize()
    res = {"out": out, "inv_rms": inv, **grads}
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in res.items()}


def run_ref(inp, eps):
    out, inv = rmsnorm.forward(inp["y"], inp["z"], inp["weight"], eps)
    return {"out": out, "inv_rms": inv, **rmsnorm.backward(inp["y"], inp["z"], inp["weight"], eps,
                                                           inp["dout"])}


CASES = [(3, 128, "f32", 1e-5), (37, 512, "f32", 0.5), (5, 256, "bf16", 1e-5),
         (200, 2048, "bf16", 1e-5), (64, 4096, "bf16", 1e-6), (1000, 384, "f32", 1e-5)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}{c[2]}")
@pytest.mark.parametrize("pass_inv", [True, False])
def test_rmsnorm_gated_every_output(case, pass_inv):
    rows, width, dtype, eps = case
    inp = synth.norm_inputs(rows, width, dtype, 7 + rows)
    gpu = run_gpu(inp, dtype, eps, pass_inv)
    ref = run_ref(inp, eps)
    errs = {k: rel_err(gpu[k], ref[k]) for k in ref}
    assert all(v <= TOL[dtype] for v in errs.values()), errs


def test_rmsnorm_gated_full_size_deterministic():
    """The SSD output of the bf16 d_inner-2048 workload (rows = B*T = 8192,
    width = H*P = 2048): every output against the oracle, and two runs equal
    bit for bit."""
    inp = synth.norm_inputs(8192, 2048, "bf16", 2048)
    a = run_gpu(inp, "bf16", 1e-5)
    b = run_gpu(inp, "bf16", 1e-5, pass_inv=False)
    c = run_gpu(inp, "bf16", 1e-5)
    ref = run_ref(inp, 1e-5)
    errs = {k: rel_err(a[k], ref[k]) for k in ref}
    print("rmsnorm full size: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
    for k in a:
        assert np.array_equal(a[k], c[k]), k
        assert np.array_equal(a[k], b[k]), k  # inv_rms recomputed inside = the forward's


def test_rmsnorm_gated_rejects_bad_width():
    import torch
    import state_space_model_analytic_gb300 as ssd
    from state_space_model_analytic_gb300 import _native as nat
    y = torch.zeros(4, 200, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(200, device="cuda")
    with pytest.raises(nat.SsdError):
        ssd.rmsnorm_gated_forward(y, y, w, 1e-5)
