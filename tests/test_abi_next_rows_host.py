"""Host-side checks of the gated RMSNorm and conv1d + SiLU entry points:
workspace sizes, and arguments rejected before anything is launched (the
library loads and validates without a GPU)."""
import ctypes
import math

import pytest

from state_space_model_analytic_gb300 import _native as nat
from state_space_model_analytic_gb300 import build as build_lib

F32, BF16 = 0, 1
FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 4)


@pytest.fixture(scope="module")
def L():
    build_lib()
    return nat.lib()


def up(v, a=256):
    return (v + a - 1) // a * a


# ---- gated RMSNorm

def test_norm_workspace_bytes(L):
    # one fp32 partial row of the weight gradient per CTA, at most 512 CTAs
    assert L.ssd_rmsnorm_gated_workspace_bytes(8192, 2048) == up(512 * 2048 * 4)
    assert L.ssd_rmsnorm_gated_workspace_bytes(1, 128) == up(512 * 128 * 4)
    assert L.ssd_rmsnorm_gated_workspace_bytes(0, 2048) == 0
    assert L.ssd_rmsnorm_gated_workspace_bytes(8, 8192) == 0


@pytest.mark.parametrize("rows,width,dtype,eps,code", [
    (0, 2048, BF16, 1e-5, nat.SSD_ERR_INVALID_ARG),      # no rows
    (8, 2048, 7, 1e-5, nat.SSD_ERR_INVALID_ARG),         # bad dtype
    (8, 300, BF16, 1e-5, nat.SSD_ERR_UNSUPPORTED),       # not a multiple of 256 (bf16)
    (8, 128, BF16, 1e-5, nat.SSD_ERR_UNSUPPORTED),       # below one 256-wide unit
    (8, 192, F32, 1e-5, nat.SSD_ERR_UNSUPPORTED),        # not a multiple of 128 (fp32)
    (8, 8192, F32, 1e-5, nat.SSD_ERR_UNSUPPORTED),       # wider than 4096
    (8, 2048, BF16, -1.0, nat.SSD_ERR_INVALID_ARG),      # negative eps
    (8, 2048, BF16, math.nan, nat.SSD_ERR_INVALID_ARG),  # NaN eps
])
def test_norm_rejects_shapes(L, rows, width, dtype, eps, code):
    rc = L.ssd_rmsnorm_gated_forward(rows, width, dtype, FAKE, FAKE, FAKE, eps, FAKE, None, None)
    assert rc == code, nat.last_error()
    rc = L.ssd_rmsnorm_gated_backward(rows, width, dtype, FAKE, FAKE, FAKE, eps, None, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, 1 << 30, None)
    assert rc == code, nat.last_error()


def test_norm_rejects_pointers_and_workspace(L):
    rc = L.ssd_rmsnorm_gated_forward(8, 2048, BF16, None, FAKE, FAKE, 1e-5, FAKE, None, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "NULL" in nat.last_error()
    rc = L.ssd_rmsnorm_gated_forward(8, 2048, BF16, MISALIGNED, FAKE, FAKE, 1e-5, FAKE, None, None)
    assert rc == nat.SSD_ERR_ALIGNMENT
    need = L.ssd_rmsnorm_gated_workspace_bytes(8, 2048)
    rc = L.ssd_rmsnorm_gated_backward(8, 2048, BF16, FAKE, FAKE, FAKE, 1e-5, None, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, need - 1, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "workspace" in nat.last_error()
    rc = L.ssd_rmsnorm_gated_backward(8, 2048, BF16, FAKE, FAKE, FAKE, 1e-5, MISALIGNED, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, need, None)
    assert rc == nat.SSD_ERR_ALIGNMENT


# ---- causal conv1d + SiLU

def test_conv_workspace_bytes(L):
    # per-CTA fp32 partials [B * ceil(T / 128)][C][K + 1] (runs of >= 16 steps,
    # 8 runs a CTA in the backward)
    assert L.ssd_conv1d_silu_workspace_bytes(4, 2048, 2304, 4) == up(4 * 16 * 2304 * 5 * 4)
    assert L.ssd_conv1d_silu_workspace_bytes(1, 5, 8, 2) == up(1 * 1 * 8 * 3 * 4)
    assert L.ssd_conv1d_silu_workspace_bytes(2, 129, 16, 1) == up(2 * 2 * 16 * 2 * 4)
    for bad in ((0, 8, 8, 4), (1, 0, 8, 4), (1, 8, 0, 4), (1, 8, 8, 0), (1, 8, 8, 5)):
        assert L.ssd_conv1d_silu_workspace_bytes(*bad) == 0, bad


@pytest.mark.parametrize("B,T,C,K,dtype,code", [
    (0, 64, 16, 4, BF16, nat.SSD_ERR_INVALID_ARG),         # no batch rows
    (70000, 64, 16, 4, BF16, nat.SSD_ERR_INVALID_ARG),     # batch above the grid limit
    (2, 1 << 30, 16, 4, BF16, nat.SSD_ERR_INVALID_ARG),    # batch * seqlen past 32-bit rows
    (1, 64, 16, 4, 7, nat.SSD_ERR_INVALID_ARG),            # bad dtype
    (1, 64, 12, 4, BF16, nat.SSD_ERR_UNSUPPORTED),         # not a multiple of 8 (bf16)
    (1, 64, 6, 4, F32, nat.SSD_ERR_UNSUPPORTED),           # not a multiple of 4 (fp32)
    (1, 64, 16, 5, BF16, nat.SSD_ERR_UNSUPPORTED),         # d_conv above 4
    (1, 64, 16, 0, BF16, nat.SSD_ERR_UNSUPPORTED),         # d_conv below 1
])
def test_conv_rejects_shapes(L, B, T, C, K, dtype, code):
    rc = L.ssd_conv1d_silu_forward(B, T, C, K, dtype, FAKE, FAKE, None, None, FAKE, None)
    assert rc == code, nat.last_error()
    rc = L.ssd_conv1d_silu_backward(B, T, C, K, dtype, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                                    None, FAKE, 1 << 40, None)
    assert rc == code, nat.last_error()


def test_conv_rejects_pointers_and_workspace(L):
    rc = L.ssd_conv1d_silu_forward(1, 64, 16, 4, BF16, None, FAKE, None, None, FAKE, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "NULL" in nat.last_error()
    rc = L.ssd_conv1d_silu_forward(1, 64, 16, 4, BF16, FAKE, FAKE, MISALIGNED, None, FAKE, None)
    assert rc == nat.SSD_ERR_ALIGNMENT
    need = L.ssd_conv1d_silu_workspace_bytes(1, 64, 16, 4)
    rc = L.ssd_conv1d_silu_backward(1, 64, 16, 4, BF16, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                                    None, FAKE, need - 1, None)
    assert rc == nat.SSD_ERR_INVALID_ARG and "workspace" in nat.last_error()
    rc = L.ssd_conv1d_silu_backward(1, 64, 16, 4, BF16, FAKE, FAKE, None, None, FAKE, None, FAKE,
                                    None, FAKE, need, None)
    assert rc == nat.SSD_ERR_INVALID_ARG
