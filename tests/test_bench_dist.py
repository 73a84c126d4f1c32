"""bench.py's multi-process path on CPU: world size 2 over gloo, each rank an
independent replica; the line reports the slowest rank's time and the tokens
of all ranks (weak scaling)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [2.0, 3.5][rank]
    ms_max, value = bench.aggregate_ranks(ms_local, 1000, dist, "cpu")
    dist.barrier()
    out[rank] = (ms_max, value)
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        ms_max, value = res[rank]
        assert ms_max == pytest.approx(3.5)
        assert value == pytest.approx(2 * 1000 / 3.5e-3)


def test_single_process_aggregation():
    sys.path.insert(0, ROOT)
    import bench
    ms_max, value = bench.aggregate_ranks(4.0, 8192)
    assert ms_max == 4.0 and value == pytest.approx(8192 / 4e-3)


def test_packed_views_are_aligned_disjoint_and_contiguous():
    """The end-to-end leg copies every input (and every output) of a step as
    one buffer: each tensor a view at a 256-byte-aligned offset, the views
    disjoint, contiguous, of the requested shape and dtype, and writes
    through a view land in the flat buffer."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    specs = {"x": ((2, 3, 4, 5), torch.bfloat16), "A": ((7,), torch.float32),
             "dt": ((2, 3, 4), torch.float32), "B": ((2, 3, 1, 16), torch.bfloat16)}
    flat, views = bench.packed(specs, "cpu")
    spans = []
    for k, (shape, dtype) in specs.items():
        v = views[k]
        assert tuple(v.shape) == shape and v.dtype == dtype and v.is_contiguous()
        off = v.data_ptr() - flat.data_ptr()
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= flat.numel()
    views["A"].fill_(2.5)
    off = views["A"].data_ptr() - flat.data_ptr()
    assert torch.equal(flat[off:off + 28].view(torch.float32), torch.full((7,), 2.5))
