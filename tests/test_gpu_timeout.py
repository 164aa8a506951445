"""Failure detection on the GPU without a fault: a bounded wait that runs out
(the library's own wait routine, on an mbarrier nothing arrives on) reports
DFLASH_ERR_TIMEOUT in the status word within its limit, and the context stays
usable for the next call."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_timeout_and_the_context_survives(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    lib.dflash_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == lib.ERR_TIMEOUT
    assert elapsed < 30.0, elapsed            # the wait is bounded (about 1 s of SM clock)
    # the context is still usable: a projection runs and is right
    x = torch.randn((17, 256), device="cuda").to(torch.bfloat16)
    w = (torch.randn((384, 256), device="cuda") / 16).to(torch.bfloat16)
    y = torch.empty((17, 384), device="cuda")
    import synth
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    ws = lib.Workspace(cfg, 16)
    lib.dflash_linear(x, w, y, ws)
    torch.cuda.synchronize()
    want = x.double() @ w.double().T
    assert (y.double() - want).abs().max().item() <= 1e-3 * want.abs().max().item() + 1e-3
