"""Host-side checks of the C ABI: the library builds for sm_103a, loads
without a GPU, exports every entry point include/ssd.h declares, and rejects
bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from state_space_model_analytic_gb300 import _native as nat
from state_space_model_analytic_gb300 import build as build_lib
from state_space_model_analytic_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_lib()
    return nat.lib()


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "ssd.h")).read()
    return re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", src)


def test_exports_every_declared_symbol(L):
    names = declared_entry_points()
    assert set(names) == set(nat.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def dims(**kw):
    base = dict(batch=2, seqlen=64, nheads=4, headdim=16, dstate=16, ngroups=2, chunk=16,
                bf16=False)
    base.update(kw)
    return nat.make_dims(**base)


def test_workspace_sizes(L):
    d = dims()
    f, b1, b2 = (L.ssd_workspace_bytes(d, w) for w in (0, 1, 2))
    states = 2 * 4 * 4 * 16 * 16 * 4
    assert f >= states and b1 >= states and b2 >= b1 + states
    # the raw-dt entry points: dt [B,T,H], A [H] and 32 x H slice sums (each
    # rounded to 256 bytes) in front
    extra = 2 * 64 * 4 * 4 + 256 + 512
    assert [L.ssd_workspace_bytes(d, w) for w in (3, 4, 5)] == [f + extra, b1 + extra, b2 + extra]
    assert L.ssd_workspace_bytes(d, 6) == 0 and L.ssd_workspace_bytes(d, -1) == 0
    for i in range(5):
        dd = synth.config_dims(i)
        d = nat.make_dims(dd.batch, dd.seqlen, dd.nheads, dd.headdim, dd.dstate, dd.ngroups,
                          dd.chunk, dd.dtype == "bf16")
        assert L.ssd_workspace_bytes(d, 0) > 0 and L.ssd_kernel_path(d) in (0, 1)


# (headdim, d_state, chunk, bf16, seqlen) -> 1: tensor-core kernels, 0: SIMT.
# The block family only: the fused bf16 kernels (headdim 64, d_state 128,
# chunk 128 or 256) also need the driver's tensor-map encoder, which a
# machine without a GPU driver lacks; the GPU tests assert their path.
@pytest.mark.parametrize("P,N,Q,bf,T,path", [
    (64, 128, 64, True, 512, 1),     # block family, d_state 128
    (64, 64, 128, False, 512, 1),    # block family, fp32 as split products
    (64, 64, 16, True, 512, 1),
    (128, 64, 64, True, 512, 1),     # block family, headdim 128
    (128, 64, 128, True, 512, 1),
    (64, 64, 256, False, 512, 1),    # chunk 256 as 128-step sub-chunks
    (64, 64, 256, True, 512, 1),
    (128, 64, 256, True, 512, 1),
    (128, 128, 64, True, 512, 1),    # headdim 128 with d_state 128
    (128, 128, 256, True, 512, 1),
    (128, 64, 64, False, 512, 0),    # headdim 128 in fp32: SIMT
    (128, 128, 64, False, 512, 0),
    (64, 128, 64, False, 512, 0),    # d_state 128 in fp32: SIMT
    (64, 64, 64, True, 192, 0),      # seqlen not a multiple of 128
    (32, 64, 64, True, 512, 0),
])
def test_kernel_path_per_shape(L, P, N, Q, bf, T, path):
    d = nat.make_dims(2, T, 4, P, N, 2, Q, bf)
    assert L.ssd_kernel_path(d) == path


@pytest.mark.parametrize("kw,code", [
    (dict(nheads=3), nat.SSD_ERR_INVALID_ARG),      # H % G
    (dict(batch=0), nat.SSD_ERR_INVALID_ARG),
    (dict(chunk=48), nat.SSD_ERR_UNSUPPORTED),
    (dict(seqlen=40), nat.SSD_ERR_UNSUPPORTED),    # T % Q
    (dict(headdim=24), nat.SSD_ERR_UNSUPPORTED),
    (dict(dstate=272), nat.SSD_ERR_UNSUPPORTED),
    (dict(headdim=128, dstate=256), nat.SSD_ERR_UNSUPPORTED),
])
def test_rejects_bad_dims(L, kw, code):
    d = dims(**kw)
    fake = ctypes.c_void_p(1 << 20)
    rc = L.ssd_forward(d, fake, fake, fake, fake, fake, fake, None, fake, None, None, fake,
                       1 << 30, None)
    assert rc == code, nat.last_error()
    assert nat.last_error()
    assert L.ssd_workspace_bytes(d, 0) == 0
    assert L.ssd_kernel_path(d) == -1


@pytest.mark.parametrize("kw,code", [
    (dict(nheads=3), nat.SSD_ERR_INVALID_ARG),
    (dict(batch=0), nat.SSD_ERR_INVALID_ARG),
    (dict(chunk=48), nat.SSD_ERR_UNSUPPORTED),
    (dict(headdim=24), nat.SSD_ERR_UNSUPPORTED),
])
def test_noalloc_rejects_bad_dims_like_ssd_forward(L, kw, code):
    d = dims(**kw)
    fake = ctypes.c_void_p(1 << 20)
    rc = L.ssd_forward_noalloc(d, fake, fake, fake, fake, fake, fake, None, fake, None, None,
                               None)
    assert rc == code, nat.last_error()
    fwd_msg = nat.last_error()
    assert fwd_msg
    rc_fwd = L.ssd_forward(d, fake, fake, fake, fake, fake, fake, None, fake, None, None, fake,
                           1 << 30, None)
    assert rc_fwd == rc and nat.last_error() == fwd_msg


def test_noalloc_rejects_fields_and_pointers_before_launching(L):
    d = dims()
    d.reserved = 1
    f = ctypes.c_void_p(1 << 20)
    assert L.ssd_forward_noalloc(d, f, f, f, f, f, f, None, f, None, None, None) == \
        nat.SSD_ERR_INVALID_ARG
    d = dims()
    d.dtype = 5
    assert L.ssd_forward_noalloc(d, f, f, f, f, f, f, None, f, None, None, None) == \
        nat.SSD_ERR_INVALID_ARG
    assert L.ssd_forward_noalloc(None, f, f, f, f, f, f, None, f, None, None, None) == \
        nat.SSD_ERR_INVALID_ARG
    d = dims()
    assert L.ssd_forward_noalloc(d, None, f, f, f, f, f, None, f, None, None, None) == \
        nat.SSD_ERR_INVALID_ARG
    bad = ctypes.c_void_p((1 << 20) + 4)
    assert L.ssd_forward_noalloc(d, f, f, f, f, f, f, None, bad, None, None, None) == \
        nat.SSD_ERR_ALIGNMENT


def test_rejects_null_misaligned_and_small_workspace(L):
    d = dims()
    f = ctypes.c_void_p(1 << 20)
    ws = L.ssd_workspace_bytes(d, 0)
    rc = L.ssd_forward(d, None, f, f, f, f, f, None, f, None, None, f, ws, None)
    assert rc == nat.SSD_ERR_INVALID_ARG
    bad = ctypes.c_void_p((1 << 20) + 4)
    rc = L.ssd_forward(d, bad, f, f, f, f, f, None, f, None, None, f, ws, None)
    assert rc == nat.SSD_ERR_ALIGNMENT
    rc = L.ssd_forward(d, f, f, f, f, f, f, None, f, None, None, ctypes.c_void_p((1 << 20) + 16),
                       ws, None)
    assert rc == nat.SSD_ERR_ALIGNMENT
    rc = L.ssd_forward(d, f, f, f, f, f, f, None, f, None, None, f, ws - 1, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "workspace" in nat.last_error()
    wsb = L.ssd_workspace_bytes(d, 1)
    rc = L.ssd_backward(d, f, f, f, f, f, f, None, f, f, f, f, f, f, f, f, None, f, wsb - 1, None)
    assert rc == nat.SSD_ERR_INVALID_ARG
    # without a history the backward needs the larger workspace
    rc = L.ssd_backward(d, f, f, f, f, f, f, None, f, None, f, f, f, f, f, f, None, f, wsb, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "recomput" in nat.last_error()
    rc = L.ssd_backward(d, f, f, f, f, f, f, None, None, f, f, f, f, f, f, f, None, f, wsb, None)
    assert rc == nat.SSD_ERR_INVALID_ARG


def test_reserved_and_dtype_fields(L):
    d = dims()
    d.reserved = 1
    assert L.ssd_workspace_bytes(d, 0) == 0
    d = dims()
    d.dtype = 7
    assert L.ssd_workspace_bytes(d, 0) == 0


def test_raw_entry_points_reject_before_launching(L):
    d = dims()
    f = ctypes.c_void_p(1 << 20)
    ws = L.ssd_workspace_bytes(d, 3)
    rc = L.ssd_forward_raw(d, f, f, None, f, f, f, f, None, f, None, None, f, ws, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "NULL" in nat.last_error()
    rc = L.ssd_forward_raw(d, f, f, f, f, f, f, f, None, f, None, None, f, ws - 1, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "workspace" in nat.last_error()
    bad = ctypes.c_void_p((1 << 20) + 8)
    rc = L.ssd_forward_raw(d, f, f, bad, f, f, f, f, None, f, None, None, f, ws, None)
    assert rc == nat.SSD_ERR_ALIGNMENT
    wsb = L.ssd_workspace_bytes(d, 4)
    args = [f] * 20
    args[7] = None  # h0
    rc = L.ssd_backward_raw(d, *args[:9], None, *args[10:18], f, wsb, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "recomput" in nat.last_error()


def test_cpu_tensors_rejected_by_front_end():
    import torch
    import state_space_model_analytic_gb300 as ssd
    x = torch.zeros(1, 16, 2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        ssd.forward(x, torch.zeros(1, 16, 2), torch.zeros(2), torch.zeros(1, 16, 1, 16),
                    torch.zeros(1, 16, 1, 16), torch.zeros(2), chunk=16)
