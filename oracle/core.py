"""ctypes wrapper around the float64 C oracle (TEST INFRASTRUCTURE ONLY).

Burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs:
``ssd_forward_state_history_reference`` (forward recurrence) and
``ssd_backward_reference`` (reverse-time backward).  All arrays are numpy
float64 in the library's layouts: x, dy [B,T,H,P]; dt [B,T,H]; A, D [H];
B, C [B,T,G,N]; h0 [B,H,P,N]; chunk history [B,nc,H,P,N].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.c_int64


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def build_oracle(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE semantics kept)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_SO)
             or os.path.getmtime(_SO) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-ffp-contract=off",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            lib.oracle_ssd_forward.restype = ctypes.c_int
            lib.oracle_ssd_forward.argtypes = [_I] * 7 + [_D] * 10 + [ctypes.c_int]
            lib.oracle_ssd_backward.restype = ctypes.c_int
            lib.oracle_ssd_backward.argtypes = [_I] * 7 + [_D] * 15 + [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return ctypes.cast(None, _D)
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _dims(x, Bm, chunk):
    Bz, T, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    return Bz, T, H, P, N, G, chunk


def ssd_forward(x, dt, A, B, C, D, h0=None, chunk=64, threads=None,
                want_y=True, want_states=True):
    """Returns (y, final_state, chunk_states); chunk_states[c] is the state
    before step c * chunk (entry 0 = h0 or zeros)."""
    x, dt, A, B, C, D, h0 = map(_f64, (x, dt, A, B, C, D, h0))
    Bz, T, H, P, N, G, Q = _dims(x, B, chunk)
    nc = -(-T // Q)
    y = np.empty_like(x) if want_y else None
    fs = np.empty((Bz, H, P, N)) if want_states else None
    cs = np.empty((Bz, nc, H, P, N)) if want_states else None
    rc = _load().oracle_ssd_forward(Bz, T, H, P, N, G, Q, _ptr(x), _ptr(dt), _ptr(A),
                                    _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(y),
                                    _ptr(fs), _ptr(cs), threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_ssd_forward failed ({rc})")
    return y, fs, cs


def ssd_backward(x, dt, A, B, C, D, h0, dy, threads=None):
    """Returns dict dx, ddt, dA, dB, dC, dD, dh0 (dh0 is zeros-shaped when
    h0 is None: the gradient w.r.t. the implicit zero initial state)."""
    x, dt, A, B, C, D, h0, dy = map(_f64, (x, dt, A, B, C, D, h0, dy))
    Bz, T, H, P, N, G, Q = _dims(x, B, 1)
    out = {
        "dx": np.empty_like(x), "ddt": np.empty_like(dt), "dA": np.empty(H),
        "dB": np.empty_like(B), "dC": np.empty_like(C), "dD": np.empty(H),
        "dh0": np.empty((Bz, H, P, N)),
    }
    rc = _load().oracle_ssd_backward(
        Bz, T, H, P, N, G, Q, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(h0), _ptr(dy), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
        _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dh0"]),
        threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_ssd_backward failed ({rc})")
    return out
