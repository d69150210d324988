"""Failure detection on the GPU without a fault: a bounded in-kernel wait that nothing satisfies gives
up after its limit, the device status word reports ENGRAM_DEVERR_TIMEOUT, and the context stays
usable for the next calls."""
import time

import pytest
import torch

import engram_conditional_memory_gb300 as ecm

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(cuda_lib):
    ecm.device_status(clear=True)
    t0 = time.perf_counter()
    ecm.check_wait_timeout(50000)  # 50 ms
    status = ecm.device_status(clear=True)
    elapsed = time.perf_counter() - t0
    assert status & ecm.DEVERR_TIMEOUT
    assert 0.04 < elapsed < 5.0
    # the context is still usable: a real call runs and reports nothing
    w = torch.rand(4096, device="cuda")
    wf = ecm.fuse_weight(w, w)
    torch.cuda.synchronize()
    assert torch.allclose(wf, w * w)
    assert ecm.device_status() == 0
