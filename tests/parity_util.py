"""Helpers for the GPU-vs-oracle parity tests.

Tolerances: max|gpu - ref| / max|ref| per output tensor (if max|ref| is 0,
max|gpu| itself); <= 1e-4 when x, B, C, dy are stored as fp32 and <= 2e-2
when they are stored as bf16 (fp32 accumulation in both cases).  The oracle
receives the storage-rounded inputs widened to float64, so the measured
error is the kernels' own.
"""
from __future__ import annotations

import numpy as np

import oracle
from state_space_model_analytic_gb300 import synth

TOL = {"f32": 1e-4, "bf16": 2e-2}
OUT_KEYS = ("y", "final_state", "chunk_states", "dx", "ddt", "dA", "dB", "dC", "dD", "dh0")


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return 0.0
    if not np.isfinite(gpu).all():
        return float("inf")
    m = np.max(np.abs(ref))
    d = np.max(np.abs(gpu - ref))
    return float(d / m) if m > 0 else float(np.max(np.abs(gpu)))


def to_device(dims: synth.Dims, inp: dict):
    import torch
    io = torch.bfloat16 if dims.dtype == "bf16" else torch.float32
    dev = torch.device("cuda", 0)

    def t(a, dtype):
        if a is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    return {"x": t(inp["x"], io), "dt": t(inp["dt"], torch.float32),
            "A": t(inp["A"], torch.float32), "B": t(inp["B"], io), "C": t(inp["C"], io),
            "D": t(inp["D"], torch.float32), "h0": t(inp["h0"], torch.float32),
            "dy": t(inp["dy"], io)}


def run_gpu(dims: synth.Dims, dev: dict, history="given"):
    """Forward then backward through the C ABI; returns numpy float64 outputs."""
    import torch
    import state_space_model_analytic_gb300 as ssd
    y, fs, cs = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                            dev["h0"], chunk=dims.chunk)
    g = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                     dev["dy"], cs if history == "given" else None, chunk=dims.chunk)
    torch.cuda.synchronize()
    out = {"y": y, "final_state": fs, "chunk_states": cs, **g}
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in out.items()}


def run_oracle(dims: synth.Dims, inp: dict, threads=None):
    y, fs, cs = oracle.ssd_forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["h0"], chunk=dims.chunk, threads=threads)
    g = oracle.ssd_backward(*(inp[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")),
                            threads=threads)
    return {"y": y, "final_state": fs, "chunk_states": cs, **g}


def group_slice(dims: synth.Dims, inp: dict, g: int):
    """The sub-problem of one group over every batch row: exact, because
    groups never interact (their own B, C and heads)."""
    hpg = dims.heads_per_group
    hs = slice(g * hpg, (g + 1) * hpg)
    sub = {"x": inp["x"][:, :, hs], "dt": inp["dt"][:, :, hs], "A": inp["A"][hs],
           "B": inp["B"][:, :, g:g + 1], "C": inp["C"][:, :, g:g + 1], "D": inp["D"][hs],
           "h0": None if inp["h0"] is None else inp["h0"][:, hs],
           "dy": inp["dy"][:, :, hs]}
    sdims = synth.Dims(dims.batch, dims.seqlen, hpg, dims.headdim, dims.dstate, 1, dims.chunk,
                       dims.dtype)
    return sdims, {k: (None if v is None else np.ascontiguousarray(v)) for k, v in sub.items()}


def slice_outputs(dims: synth.Dims, out: dict, g: int):
    hpg = dims.heads_per_group
    hs = slice(g * hpg, (g + 1) * hpg)
    return {"y": out["y"][:, :, hs], "final_state": out["final_state"][:, hs],
            "chunk_states": out["chunk_states"][:, :, hs], "dx": out["dx"][:, :, hs],
            "ddt": out["ddt"][:, :, hs], "dA": out["dA"][hs], "dB": out["dB"][:, :, g:g + 1],
            "dC": out["dC"][:, :, g:g + 1], "dD": out["dD"][hs], "dh0": out["dh0"][:, hs]}


def compare(gpu: dict, ref: dict, tol: float, keys=OUT_KEYS):
    errs = {k: rel_err(gpu[k], ref[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    return errs, bad
