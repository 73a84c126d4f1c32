"""ctypes binding to libssd_gb300.so (the C ABI of include/ssd.h).

Argument marshalling only.  Loading fails loudly when the library has not
been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

SSD_F32, SSD_BF16 = 0, 1
SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_ALIGNMENT, SSD_ERR_CUDA, \
    SSD_ERR_DEVICE_TIMEOUT = range(6)

# every entry point declared with SSD_API in include/ssd.h
EXPORTS = ("ssd_workspace_bytes", "ssd_forward", "ssd_backward", "ssd_last_error",
           "ssd_kernel_launch_count", "ssd_trace_begin", "ssd_trace_end", "ssd_trace_read",
           "ssd_trace_reset", "ssd_kernel_path", "ssd_force_kernel_path", "ssd_device_status",
           "ssd_selftest_wait_timeout", "ssd_forward_noalloc", "ssd_forward_raw",
           "ssd_backward_raw", "ssd_rmsnorm_gated_workspace_bytes", "ssd_rmsnorm_gated_forward",
           "ssd_rmsnorm_gated_backward", "ssd_conv1d_silu_workspace_bytes", "ssd_conv1d_silu_forward",
           "ssd_conv1d_silu_backward")


class SsdDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class SsdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ssd error {code}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None
_VP = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"CUDA library not built ({LIB} missing): run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(LIB)
            D = ctypes.POINTER(SsdDims)
            L.ssd_workspace_bytes.restype = ctypes.c_size_t
            L.ssd_workspace_bytes.argtypes = [D, ctypes.c_int]
            L.ssd_forward.restype = ctypes.c_int
            L.ssd_forward.argtypes = [D] + [_VP] * 11 + [ctypes.c_size_t, _VP]
            L.ssd_backward.restype = ctypes.c_int
            L.ssd_backward.argtypes = [D] + [_VP] * 17 + [ctypes.c_size_t, _VP]
            L.ssd_forward_raw.restype = ctypes.c_int
            L.ssd_forward_raw.argtypes = [D] + [_VP] * 12 + [ctypes.c_size_t, _VP]
            L.ssd_backward_raw.restype = ctypes.c_int
            L.ssd_backward_raw.argtypes = [D] + [_VP] * 19 + [ctypes.c_size_t, _VP]
            _I64, _I32, _F = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            L.ssd_rmsnorm_gated_workspace_bytes.restype = ctypes.c_size_t
            L.ssd_rmsnorm_gated_workspace_bytes.argtypes = [_I64, _I64]
            L.ssd_rmsnorm_gated_forward.restype = ctypes.c_int
            L.ssd_rmsnorm_gated_forward.argtypes = [_I64, _I64, _I32, _VP, _VP, _VP, _F, _VP,
                                                    _VP, _VP]
            L.ssd_conv1d_silu_workspace_bytes.restype = ctypes.c_size_t
            L.ssd_conv1d_silu_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
            L.ssd_conv1d_silu_forward.restype = ctypes.c_int
            L.ssd_conv1d_silu_forward.argtypes = [_I64, _I64, _I64, _I32, _I32] + [_VP] * 6
            L.ssd_conv1d_silu_backward.restype = ctypes.c_int
            L.ssd_conv1d_silu_backward.argtypes = ([_I64, _I64, _I64, _I32, _I32] + [_VP] * 9 +
                                                   [ctypes.c_size_t, _VP])
            L.ssd_rmsnorm_gated_backward.restype = ctypes.c_int
            L.ssd_rmsnorm_gated_backward.argtypes = [_I64, _I64, _I32, _VP, _VP, _VP, _F, _VP,
                                                     _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t,
                                                     _VP]
            L.ssd_last_error.restype = ctypes.c_char_p
            L.ssd_last_error.argtypes = []
            L.ssd_kernel_launch_count.restype = ctypes.c_uint64
            L.ssd_kernel_launch_count.argtypes = []
            L.ssd_kernel_path.restype = ctypes.c_int
            L.ssd_kernel_path.argtypes = [D]
            L.ssd_force_kernel_path.restype = ctypes.c_int
            L.ssd_force_kernel_path.argtypes = [ctypes.c_int]
            L.ssd_device_status.restype = ctypes.c_int
            L.ssd_device_status.argtypes = []
            L.ssd_forward_noalloc.restype = ctypes.c_int
            L.ssd_forward_noalloc.argtypes = [D] + [_VP] * 11
            L.ssd_selftest_wait_timeout.restype = ctypes.c_int
            L.ssd_selftest_wait_timeout.argtypes = [_VP]
            L.ssd_trace_begin.restype = ctypes.c_int
            L.ssd_trace_begin.argtypes = [ctypes.c_int]
            L.ssd_trace_end.restype = ctypes.c_int
            L.ssd_trace_end.argtypes = []
            L.ssd_trace_reset.restype = ctypes.c_int
            L.ssd_trace_reset.argtypes = []
            L.ssd_trace_read.restype = ctypes.c_int
            L.ssd_trace_read.argtypes = [ctypes.c_int, ctypes.c_char_p, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
            _lib = L
    return _lib


def last_error() -> str:
    return lib().ssd_last_error().decode()


def check(rc: int):
    if rc != SSD_OK:
        raise SsdError(rc, last_error())


def make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, bf16: bool) -> SsdDims:
    return SsdDims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                   SSD_BF16 if bf16 else SSD_F32, 0)


def trace_begin(capacity: int):
    check(lib().ssd_trace_begin(capacity))


def trace_end():
    check(lib().ssd_trace_end())


def trace_read() -> list[dict]:
    """Per kernel name (first-launch order): total event ms and launch count."""
    L = lib()
    out = []
    i = 0
    name = ctypes.create_string_buffer(128)
    while True:
        ms, n, un = ctypes.c_double(), ctypes.c_int(), ctypes.c_int()
        rc = L.ssd_trace_read(i, name, 128, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(un))
        if rc == SSD_ERR_INVALID_ARG:
            break
        check(rc)
        out.append({"name": name.value.decode(), "ms": ms.value, "launches": n.value,
                    "untimed": un.value})
        i += 1
    return out


def trace_reset():
    check(lib().ssd_trace_reset())
