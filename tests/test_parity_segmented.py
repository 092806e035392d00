"""The time-segmented variant of the warp-specialised scan pass against the
fp64 oracle: inside each warp the lanes split a channel's time into segments,
each segment runs the recurrence from a zero state to get its summary pair
(P, E), a warp-shuffle scan over those (Abar, Bbar x) pairs gives the state
entering every segment (eightmm.github.io "Mamba", Scan View), and the
segments run again from those states with the readout.

Selected with SSM_FORCE_SEG / SSM_FORCE_LANES; the shapes span several tiles,
a ragged tail, a partial channel block, two groups, an initial state and the
final state."""
import pytest
import torch

from parity import STATE_REL_L2, assert_close, oracle_scan, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu

VARIANTS = [(2, 2), (2, 4), (2, 8), (4, 2), (4, 4)]  # (lanes, segments)


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("lanes,seg", VARIANTS)
def test_segmented_matches_oracle(ssm, monkeypatch, io, lanes, seg):
    monkeypatch.setenv("SSM_FORCE_SEG", str(seg))
    monkeypatch.setenv("SSM_FORCE_LANES", str(lanes))
    x = I.make_scan_inputs(2, 100, 16, 776, 2, io=io, recipe="scaled", seed=60 + seg, device="cuda",
                           with_h0=True)
    y, hf = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"lanes={lanes} seg={seg}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0


@pytest.mark.parametrize("lanes,seg", [(2, 4), (4, 4)])
def test_segmented_no_gate_no_skip(ssm, monkeypatch, lanes, seg):
    """z, D and dt_bias absent, a sequence shorter than one tile."""
    monkeypatch.setenv("SSM_FORCE_SEG", str(seg))
    monkeypatch.setenv("SSM_FORCE_LANES", str(lanes))
    x = I.make_scan_inputs(1, 64, 16, 24, 1, io="bf16", recipe="unit", seed=70, device="cuda", with_z=False)
    y, hf = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C)
    torch.cuda.synchronize()
    x.D = None
    x.dt_bias = None
    ref_y, ref_h = oracle_scan(x, final_state=True)
    assert_close(to_np(y), ref_y, "bf16", "no gate")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_warp_specialised_fused_pass_of_a_chunked_plan(ssm, monkeypatch, io):
    """SSM_FUSED_KERNEL=ws runs the fused pass of a chunked plan on the
    warp-specialised kernel (each CTA a time chunk, starting from the carried
    state): y and the final state against the oracle, with an initial state."""
    monkeypatch.setenv("SSM_FUSED_KERNEL", "ws")
    monkeypatch.setenv("SSM_FORCE_CHUNKS", "5")
    x = I.make_scan_inputs(2, 192, 16, 1000, 2, io=io, recipe="scaled", seed=47, device="cuda", with_h0=True)
    assert ssm.scan_plan(2, 192, 16, 1000, 2, x.u.dtype)["chunks"] == 5
    y, hf = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"ws fused pass, 5 chunks, io={io}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0
