"""Python front end of the SSD core: torch CUDA tensors in, torch tensors out.

Torch provides device memory and the stream; every step of the forward and
backward runs in the library's CUDA kernels behind the C ABI (include/ssd.h).
Shapes: x, dy [B,T,H,P]; dt [B,T,H] fp32; A, D [H] fp32; B, C [B,T,G,N];
h0 [B,H,P,N] fp32.  x, B, C, dy share one storage type (fp32 or bf16).
"""
from __future__ import annotations

import torch

from . import _native as nat

_IO_TYPES = {torch.float32: False, torch.bfloat16: True}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


def _check(name, t, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def dims_of(x, B, chunk) -> nat.SsdDims:
    Bz, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if x.dtype not in _IO_TYPES:
        raise TypeError(f"x: unsupported dtype {x.dtype}")
    return nat.make_dims(Bz, T, H, P, N, G, chunk, _IO_TYPES[x.dtype])


def _validate_inputs(x, dt, A, B, C, D, h0, dy=None):
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    dev = x.device
    Bz, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    io = x.dtype
    _check("x", x, io, (Bz, T, H, P), dev)
    _check("dt", dt, torch.float32, (Bz, T, H), dev)
    _check("A", A, torch.float32, (H,), dev)
    _check("B", B, io, (Bz, T, G, N), dev)
    _check("C", C, io, (Bz, T, G, N), dev)
    _check("D", D, torch.float32, (H,), dev)
    if h0 is not None:
        _check("h0", h0, torch.float32, (Bz, H, P, N), dev)
    if dy is not None:
        _check("dy", dy, io, (Bz, T, H, P), dev)


def workspace_bytes(dims: nat.SsdDims, which: int) -> int:
    n = nat.lib().ssd_workspace_bytes(dims, which)
    if n == 0:
        raise nat.SsdError(nat.SSD_ERR_UNSUPPORTED, nat.last_error() or "dims rejected")
    return n


def alloc_workspace(dims: nat.SsdDims, which: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(workspace_bytes(dims, which), dtype=torch.uint8, device=device)


def kernel_path(dims: nat.SsdDims) -> int:
    return nat.lib().ssd_kernel_path(dims)


def launch_count() -> int:
    return int(nat.lib().ssd_kernel_launch_count())


def forward(x, dt, A, B, C, D, h0=None, *, chunk: int, want_final=True, want_states=True,
            out=None, workspace=None, stream=None):
    """Returns (y, final_state or None, chunk_states or None)."""
    _validate_inputs(x, dt, A, B, C, D, h0)
    dims = dims_of(x, B, chunk)
    Bz, T, H, P = x.shape
    N = B.shape[3]
    nc = T // chunk
    dev = x.device
    if out is None:
        out = {}
    y = out.get("y")
    if y is None:
        y = torch.empty_like(x)
    fs = out.get("final_state")
    if fs is None and want_final:
        fs = torch.empty(Bz, H, P, N, dtype=torch.float32, device=dev)
    cs = out.get("chunk_states")
    if cs is None and want_states:
        cs = torch.empty(Bz, nc, H, P, N, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(dims, 0, dev)
    rc = nat.lib().ssd_forward(dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                               _ptr(h0), _ptr(y), _ptr(fs), _ptr(cs), _ptr(workspace),
                               workspace.numel(), _stream_handle(stream))
    nat.check(rc)
    return y, fs, cs


def backward(x, dt, A, B, C, D, h0, dy, chunk_states=None, *, chunk: int, want_dh0=True,
             out=None, workspace=None, stream=None):
    """Gradients of sum(dy * y): dict dx, ddt, dA, dB, dC, dD, dh0 (or None)."""
    _validate_inputs(x, dt, A, B, C, D, h0, dy)
    dims = dims_of(x, B, chunk)
    Bz, T, H, P = x.shape
    N = B.shape[3]
    dev = x.device
    if chunk_states is not None:
        _check("chunk_states", chunk_states, torch.float32, (Bz, T // chunk, H, P, N), dev)
    g = dict(out) if out is not None else {}
    g.setdefault("dx", torch.empty_like(x))
    g.setdefault("ddt", torch.empty_like(dt))
    g.setdefault("dA", torch.empty_like(A))
    g.setdefault("dB", torch.empty_like(B))
    g.setdefault("dC", torch.empty_like(C))
    g.setdefault("dD", torch.empty_like(D))
    if want_dh0:
        g.setdefault("dh0", torch.empty(Bz, H, P, N, dtype=torch.float32, device=dev))
    else:
        g["dh0"] = None
    if workspace is None:
        workspace = alloc_workspace(dims, 1 if chunk_states is not None else 2, dev)
    rc = nat.lib().ssd_backward(dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(h0), _ptr(dy), _ptr(chunk_states), _ptr(g["dx"]),
                                _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                                _ptr(g["dD"]), _ptr(g["dh0"]), _ptr(workspace),
                                workspace.numel(), _stream_handle(stream))
    nat.check(rc)
    return g


def _check_raw(x, dt_raw, dt_bias, a_log):
    Bz, T, H, _ = x.shape
    dev = x.device
    _check("dt_raw", dt_raw, torch.float32, (Bz, T, H), dev)
    _check("dt_bias", dt_bias, torch.float32, (H,), dev)
    _check("a_log", a_log, torch.float32, (H,), dev)


def forward_raw(x, dt_raw, dt_bias, a_log, B, C, D, h0=None, *, chunk: int, want_final=True,
                want_states=True, out=None, workspace=None, stream=None):
    """The core with dt = softplus(dt_raw + dt_bias) and A = -exp(a_log)
    computed on the device.  Returns (y, final_state or None, chunk_states or None)."""
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    _check_raw(x, dt_raw, dt_bias, a_log)
    _validate_inputs(x, dt_raw, dt_bias, B, C, D, h0)
    dims = dims_of(x, B, chunk)
    Bz, T, H, P = x.shape
    N = B.shape[3]
    dev = x.device
    out = {} if out is None else out
    y = out.get("y")
    if y is None:
        y = torch.empty_like(x)
    fs = out.get("final_state")
    if fs is None and want_final:
        fs = torch.empty(Bz, H, P, N, dtype=torch.float32, device=dev)
    cs = out.get("chunk_states")
    if cs is None and want_states:
        cs = torch.empty(Bz, T // chunk, H, P, N, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(dims, 3, dev)
    rc = nat.lib().ssd_forward_raw(dims, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(a_log),
                                   _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(y), _ptr(fs),
                                   _ptr(cs), _ptr(workspace), workspace.numel(),
                                   _stream_handle(stream))
    nat.check(rc)
    return y, fs, cs


def backward_raw(x, dt_raw, dt_bias, a_log, B, C, D, h0, dy, chunk_states=None, *, chunk: int,
                 want_dh0=True, out=None, workspace=None, stream=None):
    """Gradients of sum(dy * y) for the raw-dt form: dict dx, d_dt_raw,
    d_dt_bias, d_a_log, dB, dC, dD, dh0 (or None)."""
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    _check_raw(x, dt_raw, dt_bias, a_log)
    _validate_inputs(x, dt_raw, dt_bias, B, C, D, h0, dy)
    dims = dims_of(x, B, chunk)
    Bz, T, H, P = x.shape
    N = B.shape[3]
    dev = x.device
    if chunk_states is not None:
        _check("chunk_states", chunk_states, torch.float32, (Bz, T // chunk, H, P, N), dev)
    g = dict(out) if out is not None else {}
    g.setdefault("dx", torch.empty_like(x))
    g.setdefault("d_dt_raw", torch.empty_like(dt_raw))
    g.setdefault("d_dt_bias", torch.empty_like(dt_bias))
    g.setdefault("d_a_log", torch.empty_like(a_log))
    g.setdefault("dB", torch.empty_like(B))
    g.setdefault("dC", torch.empty_like(C))
    g.setdefault("dD", torch.empty_like(D))
    if want_dh0:
        g.setdefault("dh0", torch.empty(Bz, H, P, N, dtype=torch.float32, device=dev))
    else:
        g["dh0"] = None
    if workspace is None:
        workspace = alloc_workspace(dims, 4 if chunk_states is not None else 5, dev)
    rc = nat.lib().ssd_backward_raw(
        dims, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(a_log), _ptr(B), _ptr(C), _ptr(D),
        _ptr(h0), _ptr(dy), _ptr(chunk_states), _ptr(g["dx"]), _ptr(g["d_dt_raw"]),
        _ptr(g["d_dt_bias"]), _ptr(g["d_a_log"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
        _ptr(g["dh0"]), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    nat.check(rc)
    return g


def rmsnorm_gated_forward(y, z, weight, eps, *, want_inv_rms=True, out=None, stream=None):
    """Gated RMSNorm over the last dimension: returns (out, inv_rms or None);
    out = y * inv_rms * weight * silu(z), inv_rms = 1 / sqrt(mean(y^2) + eps)."""
    if not y.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    width = y.shape[-1]
    rows = y.numel() // width
    if y.dtype not in _IO_TYPES:
        raise TypeError(f"y: unsupported dtype {y.dtype}")
    _check("z", z, y.dtype, tuple(y.shape), y.device)
    _check("weight", weight, torch.float32, (width,), y.device)
    if not y.is_contiguous():
        raise ValueError("y: must be contiguous")
    o = torch.empty_like(y) if out is None else out
    inv = torch.empty(y.shape[:-1], dtype=torch.float32, device=y.device) if want_inv_rms else None
    rc = nat.lib().ssd_rmsnorm_gated_forward(rows, width, int(_IO_TYPES[y.dtype]), _ptr(y), _ptr(z),
                                             _ptr(weight), float(eps), _ptr(o), _ptr(inv),
                                             _stream_handle(stream))
    nat.check(rc)
    return o, inv


def rmsnorm_gated_backward(y, z, weight, eps, dout, inv_rms=None, *, workspace=None, stream=None):
    """Gradients of sum(dout * out): dict dy, dz, dweight."""
    if not y.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    width = y.shape[-1]
    rows = y.numel() // width
    if y.dtype not in _IO_TYPES:
        raise TypeError(f"y: unsupported dtype {y.dtype}")
    for name, t in (("z", z), ("dout", dout)):
        _check(name, t, y.dtype, tuple(y.shape), y.device)
    _check("weight", weight, torch.float32, (width,), y.device)
    if inv_rms is not None:
        _check("inv_rms", inv_rms, torch.float32, tuple(y.shape[:-1]), y.device)
    g = {"dy": torch.empty_like(y), "dz": torch.empty_like(z), "dweight": torch.empty_like(weight)}
    if workspace is None:
        n = nat.lib().ssd_rmsnorm_gated_workspace_bytes(rows, width)
        if n == 0:
            raise nat.SsdError(nat.SSD_ERR_UNSUPPORTED, "width rejected")
        workspace = torch.empty(n, dtype=torch.uint8, device=y.device)
    rc = nat.lib().ssd_rmsnorm_gated_backward(
        rows, width, int(_IO_TYPES[y.dtype]), _ptr(y), _ptr(z), _ptr(weight), float(eps),
        _ptr(inv_rms), _ptr(dout), _ptr(g["dy"]), _ptr(g["dz"]), _ptr(g["dweight"]),
        _ptr(workspace), workspace.numel(), _stream_handle(stream))
    nat.check(rc)
    return g


def conv1d_silu_forward(x, weight, bias=None, init_state=None, *, out=None, stream=None):
    """Causal depthwise conv1d + SiLU over time: x [B,T,C], weight [C,K] fp32,
    bias [C] fp32, init_state [B,C,K] fp32 (None = zeros).  Returns out [B,T,C]."""
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    if x.dtype not in _IO_TYPES:
        raise TypeError(f"x: unsupported dtype {x.dtype}")
    Bz, T, C = x.shape
    K = weight.shape[1]
    _check("weight", weight, torch.float32, (C, K), x.device)
    if bias is not None:
        _check("bias", bias, torch.float32, (C,), x.device)
    if init_state is not None:
        _check("init_state", init_state, torch.float32, (Bz, C, K), x.device)
    if not x.is_contiguous():
        raise ValueError("x: must be contiguous")
    o = torch.empty_like(x) if out is None else out
    rc = nat.lib().ssd_conv1d_silu_forward(Bz, T, C, K, int(_IO_TYPES[x.dtype]), _ptr(x),
                                           _ptr(weight), _ptr(bias), _ptr(init_state), _ptr(o),
                                           _stream_handle(stream))
    nat.check(rc)
    return o


def conv1d_silu_backward(x, weight, bias, init_state, dout, *, workspace=None, stream=None):
    """Gradients of sum(dout * out): dict dx, dweight, dbias."""
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors (no CPU path exists)")
    if x.dtype not in _IO_TYPES:
        raise TypeError(f"x: unsupported dtype {x.dtype}")
    Bz, T, C = x.shape
    K = weight.shape[1]
    _check("weight", weight, torch.float32, (C, K), x.device)
    _check("dout", dout, x.dtype, (Bz, T, C), x.device)
    if bias is not None:
        _check("bias", bias, torch.float32, (C,), x.device)
    if init_state is not None:
        _check("init_state", init_state, torch.float32, (Bz, C, K), x.device)
    g = {"dx": torch.empty_like(x), "dweight": torch.empty_like(weight),
         "dbias": torch.empty(C, dtype=torch.float32, device=x.device)}
    if workspace is None:
        n = nat.lib().ssd_conv1d_silu_workspace_bytes(Bz, T, C, K)
        if n == 0:
            raise nat.SsdError(nat.SSD_ERR_UNSUPPORTED, "shape rejected")
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    rc = nat.lib().ssd_conv1d_silu_backward(
        Bz, T, C, K, int(_IO_TYPES[x.dtype]), _ptr(x), _ptr(weight), _ptr(bias), _ptr(init_state),
        _ptr(dout), _ptr(g["dx"]), _ptr(g["dweight"]), _ptr(g["dbias"]), _ptr(workspace),
        workspace.numel(), _stream_handle(stream))
    nat.check(rc)
    return g
