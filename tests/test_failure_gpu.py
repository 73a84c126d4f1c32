"""Failure detection on the GPU without a fault: a bounded device-side wait
that nothing satisfies gives up, the kernel returns, and the host reads the
timeout through ssd_device_status()."""
import time

import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_analytic_gb300 import _native as nat
    from state_space_model_analytic_gb300 import build
    build()
    L = nat.lib()
    nat.check(L.ssd_device_status())  # clear anything left over
    t0 = time.perf_counter()
    nat.check(L.ssd_selftest_wait_timeout(torch.cuda.current_stream().cuda_stream or None))
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.5 < waited < 30.0
    assert L.ssd_device_status() == nat.SSD_ERR_DEVICE_TIMEOUT
    assert "wait gave up" in nat.last_error()
    assert L.ssd_device_status() == nat.SSD_OK  # read-and-clear
    # the context is still usable
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0
