"""Writes tests/golden/modular_case.json from the float64 oracle alone.

The problem is the deterministic modular-pattern input of the parity tests on
the burn_dragon_kernel Mamba-2 backward page (``make_realistic_cuda_inputs``:
batch 1, T 32, 4 groups x 1 head, headdim 64, d_state 16, nonzero initial
state), with chunk 16.  The page prints no output values, so the stored
numbers are the oracle's; they pin later versions of the oracle (and the GPU
path) to this one.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from state_space_model_analytic_gb300 import synth  # noqa: E402

N_SAMPLES = 48


def main():
    dims, inp = synth.modular_inputs(chunk=16)
    y, fs, cs = oracle.ssd_forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                   inp["D"], inp["h0"], chunk=dims.chunk, threads=1)
    g = oracle.ssd_backward(*(inp[k] for k in ("x", "dt", "A", "B", "C", "D", "h0", "dy")),
                            threads=1)
    outs = {"y": y, "final_state": fs, "chunk_states": cs, **g}
    rng = np.random.default_rng(0)
    rec = {"dims": dims.__dict__, "samples": {}}
    for k, v in outs.items():
        flat = v.reshape(-1)
        idx = np.sort(rng.choice(flat.size, size=min(N_SAMPLES, flat.size), replace=False))
        rec["samples"][k] = {"shape": list(v.shape), "index": idx.tolist(),
                             "value": [float(f"{flat[i]:.17g}") for i in idx],
                             "sum": float(f"{flat.sum():.17g}"),
                             "absmax": float(f"{np.abs(flat).max():.17g}")}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "modular_case.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=0)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
