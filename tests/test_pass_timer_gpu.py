"""The measurement hook ssm_set_pass_timer on the GPU: with two CUDA events
registered, a chunked call (summary, carry and fused passes) and a one-pass
call each record them around their fused pass; the outputs equal those of the
same calls without the hook (the hook only records events), the elapsed time
is positive and below the whole call's, and clearing the hook stops the
recording."""
import pytest
import torch

from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


@pytest.mark.parametrize("chunks", [4, 1])
def test_pass_timer_brackets_the_fused_pass(ssm, monkeypatch, chunks):
    monkeypatch.setenv("SSM_FORCE_CHUNKS", str(chunks))
    x = I.make_scan_inputs(2, 256, 16, 4096, 1, io="bf16", recipe="scaled", seed=61, device="cuda")
    plan = ssm.scan_plan(2, 256, 16, 4096, 1, torch.bfloat16)
    assert plan["chunks"] == chunks
    y0, h0 = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()

    pb = torch.cuda.Event(enable_timing=True)
    pe = torch.cuda.Event(enable_timing=True)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    pb.record()
    pe.record()
    torch.cuda.synchronize()
    ssm.set_pass_timer(pb, pe)
    try:
        c0.record()
        y1, h1 = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
        c1.record()
        torch.cuda.synchronize()
    finally:
        ssm.set_pass_timer()
    assert torch.equal(y0, y1) and torch.equal(h0, h1)
    t_pass, t_call = pb.elapsed_time(pe), c0.elapsed_time(c1)
    assert 0.0 < t_pass <= t_call

    # Cleared: a later call leaves the events where they were.
    ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    assert pb.elapsed_time(pe) == pytest.approx(t_pass)
    assert ssm.device_status() == 0
