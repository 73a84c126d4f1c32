"""Seeded synthetic inputs for the SSD core (forward + analytic backward).

This module only draws random numbers and rounds them to the storage type the
library consumes; it holds none of the method's arithmetic.  Both the CUDA
path (through the binding) and the float64 CPU oracle take their inputs from
here, so the oracle sees exactly the values the GPU sees: tensors stored as
bf16 are rounded to bf16 first and then widened to float64, tensors stored as
fp32 are rounded to fp32.

Workload recipe (the five SSD-core workloads, numpy PCG64, seed 1000 + index,
draw order x, dt-noise, dt_bias, a_log, B, C, D, h0, dy, each drawn in
float64):

* x ~ N(0, 1)
* dt = softplus(0.5 * N(0, 1) + dt_bias[h]); dt_bias = inverse-softplus of a
  log-uniform draw in [1e-3, 0.1], one per head
* A = -exp(a_log), a_log = log U[1, 16]  (so A lies in [-16, -1])
* B, C ~ N(0, 1) / sqrt(d_state)
* D ~ U[0.5, 1.5]; dy ~ N(0, 1)
* h0 ~ N(0, 0.1^2) where the workload has an initial state, else none
* long-sequence workload: per (b, t, h) a decay r = exp(U[ln 1e-4, ln 0.999])
  is drawn in the dt-noise slot and dt = ln(r) / A_h, so exp(dt * A) spans
  1e-4 .. 0.999.

``modular_inputs`` restates the deterministic modular-pattern inputs used by
the parity tests of the burn_dragon_kernel Mamba-2 backward page
(``mod tests``, ``make_realistic_cuda_inputs``): each element is
``(idx % prime) / prime - offset`` over the flat index.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Dims", "CONFIGS", "config_dims", "make_inputs", "modular_inputs",
           "round_to"]


@dataclasses.dataclass(frozen=True)
class Dims:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str  # "f32" or "bf16": storage type of x, B, C, dy, y, dx, dB, dC

    @property
    def nchunks(self) -> int:
        return -(-self.seqlen // self.chunk)

    @property
    def heads_per_group(self) -> int:
        return self.nheads // self.ngroups

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


# name, dims, has_h0, dt draw mode
CONFIGS = {
    0: ("tiny_fp32_b1_t64_h2_p16_n16_q16",
        Dims(1, 64, 2, 16, 16, 1, 16, "f32"), False, "softplus"),
    1: ("bf16_b4_t2048_h32_p64_n128_g1_q256",
        Dims(4, 2048, 32, 64, 128, 1, 256, "bf16"), False, "softplus"),
    2: ("bf16_b2_t8192_h64_p64_n128_g8_q256",
        Dims(2, 8192, 64, 64, 128, 8, 256, "bf16"), False, "softplus"),
    3: ("fp32_h0_b8_t1024_h24_p64_n64_g1_q128",
        Dims(8, 1024, 24, 64, 64, 1, 128, "f32"), True, "softplus"),
    4: ("bf16_h0_long_b1_t32768_h32_p64_n128_g4_q256",
        Dims(1, 32768, 32, 64, 128, 4, 256, "bf16"), True, "decay_span"),
}


def config_dims(idx: int) -> Dims:
    return CONFIGS[idx][1]


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage type and widen back to float64."""
    a = np.asarray(a, dtype=np.float64)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        return t.to(torch.bfloat16).to(torch.float64).numpy()
    raise ValueError(dtype)


def _softplus(v):
    return np.logaddexp(0.0, v)


def _inv_softplus(v):
    return np.log(np.expm1(v))


def make_inputs(dims: Dims, seed: int, has_h0: bool, dt_mode: str = "softplus",
                with_dy: bool = True) -> dict:
    """Draw one problem.  Returns float64 arrays holding storage-rounded values.

    Keys: x [B,T,H,P], dt [B,T,H], A [H], B [B,T,G,N], C [B,T,G,N], D [H],
    h0 [B,H,P,N] or None, dy [B,T,H,P]; and the raw parameters the dt and A
    are drawn through: dt_raw [B,T,H] (None for "decay_span"), dt_bias [H],
    a_log [H].
    """
    d = dims
    rng = np.random.Generator(np.random.PCG64(seed))
    Bz, T, H, P, N, G = d.batch, d.seqlen, d.nheads, d.headdim, d.dstate, d.ngroups
    x = rng.standard_normal((Bz, T, H, P))
    if dt_mode == "decay_span":
        noise = rng.uniform(math.log(1e-4), math.log(0.999), size=(Bz, T, H))
    else:
        noise = rng.standard_normal((Bz, T, H))
    dt_bias = _inv_softplus(np.exp(rng.uniform(math.log(1e-3), math.log(0.1),
                                               size=(H,))))
    a_log = np.log(rng.uniform(1.0, 16.0, size=(H,)))
    Bm = rng.standard_normal((Bz, T, G, N)) / math.sqrt(N)
    Cm = rng.standard_normal((Bz, T, G, N)) / math.sqrt(N)
    D = rng.uniform(0.5, 1.5, size=(H,))
    h0 = rng.standard_normal((Bz, H, P, N)) * 0.1 if has_h0 else None
    dy = rng.standard_normal((Bz, T, H, P)) if with_dy else None

    A = round_to(-np.exp(a_log), "f32")
    if dt_mode == "decay_span":
        # noise holds ln(r); dt = ln(r) / A_h is positive because A_h < 0
        dt = noise / A[None, None, :]
    else:
        dt = _softplus(0.5 * noise + dt_bias[None, None, :])
    io = d.dtype
    return {
        "x": round_to(x, io),
        "dt": round_to(dt, "f32"),
        "A": A,
        "B": round_to(Bm, io),
        "C": round_to(Cm, io),
        "D": round_to(D, "f32"),
        "h0": None if h0 is None else round_to(h0, "f32"),
        "dy": None if dy is None else round_to(dy, io),
        "dt_raw": None if dt_mode == "decay_span" else round_to(0.5 * noise, "f32"),
        "dt_bias": round_to(dt_bias, "f32"),
        "a_log": round_to(a_log, "f32"),
    }


def config_inputs(idx: int, with_dy: bool = True) -> tuple[Dims, dict]:
    _, dims, has_h0, mode = CONFIGS[idx]
    return dims, make_inputs(dims, 1000 + idx, has_h0, mode, with_dy)


def modular_inputs(chunk: int = 16) -> tuple[Dims, dict]:
    """Deterministic modular-pattern problem: batch 1, T 32, 4 groups of one
    head each, headdim 64, d_state 16, with an initial state (fp32)."""
    Bz, T, G, hpg, P, N = 1, 32, 4, 1, 64, 16
    H = G * hpg

    def pat(count, prime, offset):
        idx = np.arange(count, dtype=np.int64)
        return (idx % prime).astype(np.float64) / prime + offset

    x = pat(Bz * T * H * P, 257, -0.5).reshape(Bz, T, H, P)
    Bm = pat(Bz * T * G * N, 263, -0.5).reshape(Bz, T, G, N)
    Cm = pat(Bz * T * G * N, 269, -0.5).reshape(Bz, T, G, N)
    dt = pat(Bz * T * H, 271, 0.05).reshape(Bz, T, H)
    a_log = pat(H, 277, -0.25)
    D = pat(H, 281, -0.25)
    h0 = pat(Bz * H * P * N, 283, -0.5).reshape(Bz, H, P, N)
    dy = pat(Bz * T * H * P, 293, -0.5).reshape(Bz, T, H, P)
    dims = Dims(Bz, T, H, P, N, G, chunk, "f32")
    f = lambda a: round_to(a, "f32")
    return dims, {"x": f(x), "dt": f(dt), "A": f(-np.exp(a_log)), "B": f(Bm),
                  "C": f(Cm), "D": f(D), "h0": f(h0), "dy": f(dy)}


def norm_inputs(rows: int, width: int, dtype: str, seed: int) -> dict:
    """Gated-RMSNorm inputs: y, z, dout ~ N(0, 1) [rows, width] rounded to the
    storage type; weight ~ U[0.5, 1.5] [width] fp32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    y = rng.standard_normal((rows, width))
    z = rng.standard_normal((rows, width))
    w = rng.uniform(0.5, 1.5, size=(width,))
    g = rng.standard_normal((rows, width))
    return {"y": round_to(y, dtype), "z": round_to(z, dtype), "weight": round_to(w, "f32"),
            "dout": round_to(g, dtype)}


def conv_inputs(batch: int, seqlen: int, channels: int, d_conv: int, dtype: str, seed: int,
                with_init: bool = True) -> dict:
    """Conv1d + SiLU inputs: x, dout ~ N(0, 1) [B, T, C] rounded to the storage
    type; weight ~ N(0, 1) / sqrt(d_conv) [C, K]; bias ~ N(0, 0.1^2) [C];
    init_state ~ N(0, 1) [B, C, K] or None; all but x, dout fp32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((batch, seqlen, channels))
    w = rng.standard_normal((channels, d_conv)) / math.sqrt(d_conv)
    b = rng.standard_normal(channels) * 0.1
    init = rng.standard_normal((batch, channels, d_conv)) if with_init else None
    g = rng.standard_normal((batch, seqlen, channels))
    return {"x": round_to(x, dtype), "weight": round_to(w, "f32"), "bias": round_to(b, "f32"),
            "init_state": None if init is None else round_to(init, "f32"),
            "dout": round_to(g, dtype)}
