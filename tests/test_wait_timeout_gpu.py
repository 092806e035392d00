"""Failure detection of the bounded device-side waits, on the GPU, without a
GPU fault: the producer warp of the warp-specialised scan pass is told to
stop issuing loads at one tile (a flag nothing else sets), so the consumer
warps' waits for that tile run out.  With a 1 ms budget each wait gives up,
records the timeout in the library's device error word and in the caller's
workspace status word, and the kernel returns; the producer has waited for
every load it issued, so nothing is left in flight.  The host reads
SSM_ERR_TIMEOUT from both, and the context stays usable: the next call,
without the flag, matches the oracle."""
import time

import pytest
import torch

from parity import assert_close, oracle_scan, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu

SSM_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def test_wait_that_runs_out_is_reported_and_the_context_survives(ssm, monkeypatch):
    monkeypatch.setenv("SSM_FORCE_CHUNKS", "1")  # one pass: the warp-specialised kernel
    x = I.make_scan_inputs(2, 256, 16, 320, 1, io="bf16", seed=95, device="cuda")  # 20 tiles of 16 steps
    plan = ssm.scan_plan(2, 256, 16, 320, 1, torch.bfloat16)
    assert plan["chunks"] == 1 and plan["staged"]
    ws = ssm.alloc_workspace(ssm.chunked_workspace_size(2, 256, 16, 320, 1, torch.bfloat16), "cuda")
    assert ssm.device_status(clear=True) == 0

    monkeypatch.setenv("SSM_DEBUG_STOP_LOADS_AT_TILE", "5")
    monkeypatch.setenv("SSM_DEBUG_WAIT_BUDGET_US", "1000")
    t0 = time.time()
    ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, workspace=ws)
    assert ssm.workspace_status(ws) == SSM_ERR_TIMEOUT
    assert ssm.device_status(clear=True) == SSM_ERR_TIMEOUT
    assert time.time() - t0 < 30.0

    monkeypatch.delenv("SSM_DEBUG_STOP_LOADS_AT_TILE")
    monkeypatch.delenv("SSM_DEBUG_WAIT_BUDGET_US")
    y, _ = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, workspace=ws)
    torch.cuda.synchronize()
    assert ssm.workspace_status(ws) == 0
    assert ssm.device_status() == 0
    assert_close(to_np(y), oracle_scan(x), "bf16", "after a timeout")
