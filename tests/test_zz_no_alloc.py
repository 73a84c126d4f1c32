"""ssd_forward_noalloc: the forward for callers that cannot allocate device
memory (a host framework that owns every byte through its own pool, a
latency-critical path where an allocation may synchronise the device or run
out of memory).  It works in a fixed scratch array inside the library
instead of a caller workspace.

Checked through the C ABI against ssd_forward on the same inputs, on two
calls in a row (the shared scratch keeps the previous call's contents), with
and without a caller history buffer, on every kernel sequence the forward
has (single-pass tensor-core, unfused tensor-core, d_state-64 tensor-core
on blocks and on sub-chunks, SIMT): the launch sequence
is ssd_forward's, so the outputs must be bit-for-bit equal.  One case is also
compared with the float64 oracle.  Oversized problems are refused before
anything is launched.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from state_space_model_analytic_gb300 import synth

from parity_util import TOL, rel_err, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import _native as nat
    from state_space_model_analytic_gb300 import build
    build()
    return nat


CASES = [
    synth.Dims(4, 256, 32, 64, 128, 1, 256, "bf16"),   # single-pass tensor-core forward
    synth.Dims(2, 1024, 4, 64, 128, 2, 256, "bf16"),  # unfused tensor-core kernels
    synth.Dims(2, 512, 4, 64, 64, 2, 64, "f32"),      # d_state-64 tensor-core kernels
    synth.Dims(1, 512, 4, 64, 64, 1, 256, "f32"),     # the same on 128-step sub-chunks
    synth.Dims(1, 256, 3, 32, 48, 1, 64, "f32"),       # SIMT kernels
]


def _noalloc(nat, dims, dev, with_history, fs_like, cs_like):
    import torch
    cd = nat.make_dims(dims.batch, dims.seqlen, dims.nheads, dims.headdim, dims.dstate,
                       dims.ngroups, dims.chunk, dims.dtype == "bf16")
    stream = torch.cuda.current_stream().cuda_stream or None
    y = torch.full_like(dev["x"], float("nan"))
    fs = torch.full_like(fs_like, float("nan"))
    cs = torch.full_like(cs_like, float("nan")) if with_history else None
    rc = nat.lib().ssd_forward_noalloc(
        cd, _ptr(dev["x"]), _ptr(dev["dt"]), _ptr(dev["A"]), _ptr(dev["B"]), _ptr(dev["C"]),
        _ptr(dev["D"]), _ptr(dev["h0"]), _ptr(y), _ptr(fs), _ptr(cs), stream)
    assert rc == nat.SSD_OK, nat.last_error()
    torch.cuda.synchronize()
    return y, fs, cs


@pytest.mark.parametrize("dims", CASES, ids=lambda d: f"{d.dtype}_b{d.batch}_h{d.nheads}")
@pytest.mark.parametrize("with_history", [True, False])
def test_noalloc_forward_equals_workspace_forward(lib, dims, with_history):
    import torch
    import state_space_model_analytic_gb300 as ssd
    nat = lib
    inp = synth.make_inputs(dims, 99, True, "softplus")
    dev = to_device(dims, inp)
    y_ref, fs_ref, cs_ref = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"],
                                        dev["D"], dev["h0"], chunk=dims.chunk)
    torch.cuda.synchronize()
    for call in range(2):
        y, fs, cs = _noalloc(nat, dims, dev, with_history, fs_ref, cs_ref)
        assert torch.equal(y, y_ref), f"call {call}: y"
        assert torch.equal(fs, fs_ref), f"call {call}: final state"
        if with_history:
            assert torch.equal(cs, cs_ref), f"call {call}: chunk states"


def test_noalloc_forward_matches_oracle(lib):
    nat = lib
    dims = CASES[0]
    inp = synth.make_inputs(dims, 7, True, "softplus")
    dev = to_device(dims, inp)
    ref = run_oracle(dims, inp)
    import torch
    fs_like = torch.empty(dims.batch, dims.nheads, dims.headdim, dims.dstate, device="cuda")
    cs_like = torch.empty(dims.batch, dims.nchunks, dims.nheads, dims.headdim, dims.dstate,
                          device="cuda")
    y, fs, cs = _noalloc(nat, dims, dev, True, fs_like, cs_like)
    for name, got in (("y", y), ("final_state", fs), ("chunk_states", cs)):
        e = rel_err(got.float().cpu().numpy(), ref[name])
        assert e <= TOL[dims.dtype], (name, e)


def test_noalloc_refuses_what_does_not_fit(lib):
    import torch
    nat = lib
    # chunk states of this problem (B*nc*H*P*N floats = 16 MiB) exceed the scratch
    cd = nat.make_dims(2, 4096, 8, 64, 128, 1, 128, True)
    buf = torch.zeros(64, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    rc = nat.lib().ssd_forward_noalloc(cd, p, p, p, p, p, p, None, p, None, None, None)
    assert rc == nat.SSD_ERR_UNSUPPORTED
    assert "scratch" in nat.last_error()
