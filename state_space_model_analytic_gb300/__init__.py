"""Mamba-2 SSD core (forward + analytic backward) on GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind a C ABI
(include/ssd.h, library ``_build/libssd_gb300.so``); this package is the
build step, a ctypes binding and a thin torch front end.  Importing it does
not load the library; the first call does, and fails loudly when the
library is missing.
"""
from .build import build  # noqa: F401

__all__ = ["build", "forward", "backward", "forward_raw", "backward_raw",
           "rmsnorm_gated_forward", "rmsnorm_gated_backward", "conv1d_silu_forward",
           "conv1d_silu_backward", "workspace_bytes", "kernel_path", "launch_count"]


def __getattr__(name):
    if name in ("forward", "backward", "forward_raw", "backward_raw", "rmsnorm_gated_forward",
                "rmsnorm_gated_backward", "conv1d_silu_forward", "conv1d_silu_backward",
                "workspace_bytes", "kernel_path", "launch_count", "alloc_workspace", "dims_of"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
