"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small problems are compared element by element on every output; the five
SSD-core workloads are run at full size in the same launch configuration as
the benchmark and compared on one whole group (all batch rows, every head of
the group), which the oracle computes exactly because groups are
independent.
"""
import numpy as np
import pytest

from state_space_model_analytic_gb300 import synth

from parity_util import (TOL, compare, group_slice, rel_err, run_gpu, run_oracle,
                         slice_outputs, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import build
    build()


def check_problem(dims, inp, history="given"):
    gpu = run_gpu(dims, to_device(dims, inp), history)
    ref = run_oracle(dims, inp)
    errs, bad = compare(gpu, ref, TOL[dims.dtype])
    assert not bad, f"{dims}: {errs}"
    return errs


SMALL = [
    # (B, T, H, P, N, G, Q, dtype, h0, mode)
    (1, 64, 2, 16, 16, 1, 16, "f32", False, "softplus"),
    (2, 96, 4, 32, 16, 2, 32, "f32", True, "softplus"),
    (1, 128, 3, 16, 48, 3, 64, "f32", True, "softplus"),
    (2, 256, 2, 64, 64, 1, 128, "f32", True, "softplus"),
    (1, 512, 2, 64, 128, 2, 256, "f32", True, "decay_span"),
    (1, 256, 4, 64, 128, 1, 256, "bf16", False, "softplus"),
    (2, 512, 4, 64, 128, 2, 256, "bf16", True, "decay_span"),
    (1, 256, 2, 128, 128, 1, 128, "f32", True, "softplus"),
    (1, 128, 2, 64, 256, 1, 64, "bf16", True, "softplus"),
    (1, 32, 8, 16, 32, 8, 32, "f32", True, "softplus"),  # one chunk, G = H
    (1, 384, 2, 64, 128, 1, 128, "bf16", True, "decay_span"),
    (2, 256, 6, 64, 128, 3, 128, "bf16", False, "softplus"),
    (1, 128, 2, 64, 128, 2, 128, "bf16", True, "softplus"),  # one chunk
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c[:7])) + c[7])
def test_small_problems_every_output(case):
    Bz, T, H, P, N, G, Q, dt_, h0, mode = case
    dims = synth.Dims(Bz, T, H, P, N, G, Q, dt_)
    inp = synth.make_inputs(dims, 7 + T + H, h0, mode)
    check_problem(dims, inp)


def test_modular_case_and_recompute_mode():
    dims, inp = synth.modular_inputs(chunk=16)
    e1 = check_problem(dims, inp, "given")
    e2 = check_problem(dims, inp, "recompute")
    assert e1 == e2


def test_tiny_workload_config0_every_output():
    dims, inp = synth.config_inputs(0)
    check_problem(dims, inp)


def test_history_given_or_recomputed_is_bitwise_equal_and_deterministic():
    dims = synth.Dims(2, 512, 4, 64, 128, 2, 128, "bf16")
    inp = synth.make_inputs(dims, 3, True, "softplus")
    dev = to_device(dims, inp)
    a = run_gpu(dims, dev, "given")
    b = run_gpu(dims, dev, "recompute")
    c = run_gpu(dims, dev, "given")
    for k in a:
        assert np.array_equal(a[k], b[k]), k
        assert np.array_equal(a[k], c[k]), k


def test_chunk_size_invariance():
    base = synth.Dims(1, 512, 2, 64, 64, 1, 64, "f32")
    inp = synth.make_inputs(base, 5, True, "softplus")
    outs = {}
    for q in (32, 64, 128, 256):
        d = synth.Dims(1, 512, 2, 64, 64, 1, q, "f32")
        outs[q] = run_gpu(d, to_device(d, inp))
    for q in (32, 128, 256):
        for k in ("y", "final_state", "dx", "ddt", "dA", "dB", "dC", "dD", "dh0"):
            assert rel_err(outs[q][k], outs[64][k]) < 1e-4, (q, k)
        # history at a coarser chunk is a subsample of the finer one
    np.testing.assert_allclose(outs[128]["chunk_states"], outs[64]["chunk_states"][:, ::2],
                               rtol=0, atol=1e-4 * np.abs(outs[64]["chunk_states"]).max())


def test_A_zero_no_decay():
    dims = synth.Dims(1, 256, 2, 32, 32, 1, 64, "f32")
    inp = synth.make_inputs(dims, 9, True, "softplus")
    inp["A"] = np.zeros_like(inp["A"])
    check_problem(dims, inp)


def test_outputs_stay_inside_their_buffers():
    """Canary words after every output survive a forward + backward."""
    import torch
    import state_space_model_analytic_gb300 as ssd
    dims = synth.Dims(1, 96, 3, 16, 32, 1, 32, "f32")
    inp = synth.make_inputs(dims, 4, True, "softplus")
    dev = to_device(dims, inp)
    pad = 64
    canary = -12345.0

    def padded(shape, dtype=torch.float32):
        n = int(np.prod(shape))
        buf = torch.full((n + pad,), canary, dtype=dtype, device="cuda")
        return buf, buf[:n].view(*shape)

    bufs = {}
    Bz, T, H, P, N, G, Q = 1, 96, 3, 16, 32, 1, 32
    shapes = {"y": (Bz, T, H, P), "final_state": (Bz, H, P, N), "chunk_states": (Bz, T // Q, H, P, N),
              "dx": (Bz, T, H, P), "ddt": (Bz, T, H), "dA": (H,), "dB": (Bz, T, G, N),
              "dC": (Bz, T, G, N), "dD": (H,), "dh0": (Bz, H, P, N)}
    views = {}
    for k, s in shapes.items():
        bufs[k], views[k] = padded(s)
    y, fs, cs = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                            chunk=Q, out={"y": views["y"], "final_state": views["final_state"],
                                          "chunk_states": views["chunk_states"]})
    ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"], dev["dy"],
                 cs, chunk=Q, out={k: views[k] for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dh0")})
    torch.cuda.synchronize()
    for k, b in bufs.items():
        tail = b[-pad:].cpu().numpy()
        assert (tail == canary).all(), k


FULL = [1, 2, 3, 4]


@pytest.mark.parametrize("idx", FULL)
def test_full_size_workload_one_group(idx):
    """Full-size workload, benchmark launch configuration; the oracle
    computes one whole group (last group) over every batch row."""
    dims, inp = synth.config_inputs(idx)
    gpu = run_gpu(dims, to_device(dims, inp))
    g = dims.ngroups - 1
    sdims, sub = group_slice(dims, inp, g)
    ref = run_oracle(sdims, sub)
    errs, bad = compare(slice_outputs(dims, gpu, g), ref, TOL[dims.dtype])
    print(f"config {idx}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert not bad, errs
    for v in gpu.values():
        assert np.isfinite(v).all()


@pytest.mark.parametrize("q,h0", [(128, True), (256, True), (128, False)])
def test_single_pass_forward_look_back(q, h0):
    """Shapes with enough (b, h) pairs for the single-pass forward, whose CTAs
    pass chunk-end states to the next chunk through the history (look-back):
    it must be the kernel that ran; one group against the oracle; every
    output against the SIMT path (forced); y and the states bit for bit on a
    second run."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(4, 1024, 64, 64, 128, 16, q, "bf16")  # B * H = 256 (b, h) pairs
    inp = synth.make_inputs(dims, 29, h0, "softplus")
    dev = to_device(dims, inp)
    nat.trace_begin(64)
    try:
        tc = run_gpu(dims, dev)
    finally:
        nat.trace_end()
    names = [r["name"] for r in nat.trace_read()]
    nat.trace_reset()
    assert "fwd_single_tc" in names, names
    again = run_gpu(dims, dev)
    for k in ("y", "final_state", "chunk_states"):
        assert np.array_equal(tc[k], again[k]), k
    g = dims.ngroups - 1
    sdims, sub = group_slice(dims, inp, g)
    errs, bad = compare(slice_outputs(dims, tc, g), run_oracle(sdims, sub), TOL["bf16"])
    assert not bad, errs
    nat.check(nat.lib().ssd_force_kernel_path(0))
    try:
        simt = run_gpu(dims, dev)
    finally:
        nat.check(nat.lib().ssd_force_kernel_path(-1))
    for k in tc:
        assert rel_err(tc[k], simt[k]) < TOL["bf16"], k
    nat.check(nat.lib().ssd_device_status())


@pytest.mark.parametrize("q", [128, 256])
def test_tensor_core_and_simt_paths_agree(q):
    """The tcgen05 path and the SIMT path (forced) give the same results
    within the bf16 tolerance, and both match the oracle."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(2, 512, 4, 64, 128, 2, q, "bf16")
    inp = synth.make_inputs(dims, 21, True, "softplus")
    dev = to_device(dims, inp)
    assert nat.lib().ssd_kernel_path(nat.make_dims(2, 512, 4, 64, 128, 2, q, True)) == 1
    tc = run_gpu(dims, dev)
    nat.check(nat.lib().ssd_force_kernel_path(0))
    try:
        simt = run_gpu(dims, dev)
    finally:
        nat.check(nat.lib().ssd_force_kernel_path(-1))
    ref = run_oracle(dims, inp)
    for k in tc:
        assert rel_err(tc[k], ref[k]) < TOL["bf16"], k
        assert rel_err(simt[k], ref[k]) < TOL["bf16"], k
        assert rel_err(tc[k], simt[k]) < TOL["bf16"], k
    nat.check(nat.lib().ssd_device_status())


def test_graph_replay_and_side_stream_match_eager_bitwise():
    """The forward + backward API calls captured in a CUDA graph (as the
    benchmark replays them) and the same calls on a side stream give the
    eager results bit for bit, on the tensor-core path."""
    import torch
    import state_space_model_analytic_gb300 as ssd
    dims = synth.Dims(2, 1024, 8, 64, 128, 2, 256, "bf16")
    inp = synth.make_inputs(dims, 17, True, "softplus")
    dev = to_device(dims, inp)
    Q = dims.chunk
    cd = ssd.dims_of(dev["x"], dev["B"], Q)
    ws_f = ssd.alloc_workspace(cd, 0, dev["x"].device)
    ws_b = ssd.alloc_workspace(cd, 1, dev["x"].device)

    def buffers():
        y = torch.empty_like(dev["x"])
        fo = {"y": y, "final_state": torch.empty_like(dev["h0"]),
              "chunk_states": torch.empty(2, 1024 // Q, 8, 64, 128, device="cuda")}
        bo = {"dx": torch.empty_like(dev["x"]), "ddt": torch.empty_like(dev["dt"]),
              "dA": torch.empty_like(dev["A"]), "dB": torch.empty_like(dev["B"]),
              "dC": torch.empty_like(dev["C"]), "dD": torch.empty_like(dev["D"]),
              "dh0": torch.empty_like(dev["h0"])}
        return fo, bo

    def step(fo, bo):
        ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                    chunk=Q, out=fo, workspace=ws_f)
        ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                     dev["dy"], fo["chunk_states"], chunk=Q, out=bo, workspace=ws_b)

    ref_f, ref_b = buffers()
    step(ref_f, ref_b)
    torch.cuda.synchronize()

    g_f, g_b = buffers()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(g_f, g_b)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()

    s_f, s_b = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(s_f, s_b)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for name, ref in list(ref_f.items()) + list(ref_b.items()):
        other_g = g_f.get(name, g_b.get(name))
        other_s = s_f.get(name, s_b.get(name))
        assert torch.equal(ref, other_g), name
        assert torch.equal(ref, other_s), name


@pytest.mark.parametrize("q", [128, 256])
def test_optional_outputs_absent_on_tensor_core_path(q):
    """No final state, no returned history (the forward keeps it in its
    workspace) and no dh0: the outputs that remain match the full call."""
    import torch
    import state_space_model_analytic_gb300 as ssd
    dims = synth.Dims(1, 512, 8, 64, 128, 1, q, "bf16")
    inp = synth.make_inputs(dims, 23, True, "softplus")
    dev = to_device(dims, inp)
    y, fs, cs = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                            dev["h0"], chunk=q)
    g = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                     dev["dy"], cs, chunk=q)
    y2, fs2, cs2 = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                               dev["h0"], chunk=q, want_final=False, want_states=False)
    g2 = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                      dev["dy"], None, chunk=q, want_dh0=False)
    torch.cuda.synchronize()
    assert fs2 is None and cs2 is None and g2["dh0"] is None
    assert torch.equal(y, y2)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        assert torch.equal(g[k], g2[k]), k


@pytest.mark.parametrize("shape", [(2, 1024, 8, 64, 128, 4, 256), (1, 2048, 64, 64, 128, 16, 256),
                                   (3, 768, 12, 64, 128, 3, 128)])
def test_repeated_steps_are_bitwise_identical(shape):
    """Twenty forward + backward steps on one input give the first step's
    outputs bit for bit: the backward's split units (arrival tickets,
    written-partial counters, the last segment summing in segment order)
    and the single-pass forward's tile claims leave no run-to-run variation.
    Shapes with small head groups, so that most units are split over CTAs;
    the second fills the GPU's fused state scans and single-pass forward."""
    import torch
    import state_space_model_analytic_gb300 as ssd
    dims = synth.Dims(*shape, "bf16")
    inp = synth.make_inputs(dims, 31, True, "softplus")
    dev = to_device(dims, inp)
    ref = None
    for _ in range(20):
        y, fs, cs = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                dev["h0"], chunk=dims.chunk)
        g = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                         dev["dy"], cs, chunk=dims.chunk)
        out = {"y": y, "final_state": fs, "chunk_states": cs, **g}
        if ref is None:
            ref = {k: v.clone() for k, v in out.items() if v is not None}
            continue
        for k, v in ref.items():
            assert torch.equal(out[k], v), k
    torch.cuda.synchronize()


def test_fused_paths_with_decay_span_inputs():
    """The single-pass forward and the backward whose state scan writes the
    mid-chunk state gradients (g_mid, 256-step chunks taken in two halves)
    on decay-span inputs (decays down to 1e-4 within a chunk, where the
    halves' weights exp(cs_i - cs_127) and the regrouped recurrence matter),
    with h0: one group against the oracle, every output."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(4, 1024, 64, 64, 128, 16, 256, "bf16")  # B * H = 256: fused kernels
    inp = synth.make_inputs(dims, 37, True, "decay_span")
    dev = to_device(dims, inp)
    nat.trace_begin(64)
    try:
        gpu = run_gpu(dims, dev)
    finally:
        nat.trace_end()
    names = [r["name"] for r in nat.trace_read()]
    nat.trace_reset()
    assert "fwd_single_tc" in names and "state_scan_bwd_tc" in names, names
    g = 5
    sdims, sub = group_slice(dims, inp, g)
    errs, bad = compare(slice_outputs(dims, gpu, g), run_oracle(sdims, sub), TOL["bf16"])
    print(", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert not bad, errs
    nat.check(nat.lib().ssd_device_status())


def test_recompute_mode_on_fused_kernels():
    """The backward without a history on a shape that fills the GPU with the
    fused kernels: it recomputes the chunk-start states with the forward
    state scan, then runs the state scan that writes g_mid and the
    tensor-core backward.  Against the oracle (one group, every gradient)
    and against the history-given call (its history came from the
    single-pass forward, so the two agree within the tolerance, not bit
    for bit)."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(4, 1024, 64, 64, 128, 16, 256, "bf16")  # B * H = 256
    inp = synth.make_inputs(dims, 41, True, "softplus")
    dev = to_device(dims, inp)
    nat.trace_begin(64)
    try:
        rec = run_gpu(dims, dev, "recompute")
    finally:
        nat.trace_end()
    names = [r["name"] for r in nat.trace_read()]
    nat.trace_reset()
    assert "state_scan_fwd_tc" in names and "state_scan_bwd_tc" in names, names
    given = run_gpu(dims, dev, "given")
    g = 11
    sdims, sub = group_slice(dims, inp, g)
    keys = ("dx", "ddt", "dA", "dB", "dC", "dD", "dh0")
    errs, bad = compare(slice_outputs(dims, rec, g), run_oracle(sdims, sub), TOL["bf16"], keys)
    assert not bad, errs
    for k in keys:
        assert rel_err(rec[k], given[k]) < TOL["bf16"], k
    nat.check(nat.lib().ssd_device_status())


@pytest.mark.parametrize("shape", [(2, 256, 64, 64, 128, 8, 256),    # one chunk, 128 tiles
                                   (1, 512, 128, 64, 128, 32, 256),  # two chunks, 256 tiles
                                   (4, 256, 32, 64, 128, 4, 128)])   # two chunks of 128
def test_single_pass_forward_few_tiles(shape):
    """The single-pass forward's resident CTAs when the tiles number fewer
    than two per SM (some CTAs take one tile or none) and sequences have one
    or two chunks (no look-back, or one hop): it must be that kernel; one
    group against the oracle, every output."""
    from state_space_model_analytic_gb300 import _native as nat
    dims = synth.Dims(*shape, "bf16")
    inp = synth.make_inputs(dims, 43, True, "softplus")
    dev = to_device(dims, inp)
    nat.trace_begin(64)
    try:
        gpu = run_gpu(dims, dev)
    finally:
        nat.trace_end()
    names = [r["name"] for r in nat.trace_read()]
    nat.trace_reset()
    assert "fwd_single_tc" in names, names
    g = dims.ngroups - 1
    sdims, sub = group_slice(dims, inp, g)
    errs, bad = compare(slice_outputs(dims, gpu, g), run_oracle(sdims, sub), TOL["bf16"])
    assert not bad, errs
    nat.check(nat.lib().ssd_device_status())
