"""GPU parity of the TMA-staged scan path (rows whose byte length is a multiple
of 16) against the fp64 oracle: every lanes-per-channel variant, single pass
and time-chunked with carried summaries, ragged time tails, partial channel
blocks, several groups, and writes confined to y."""
import os

import numpy as np
import pytest
import torch

from parity import STATE_REL_L2, assert_close, oracle_scan, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


@pytest.fixture
def env():
    saved = {k: os.environ.get(k) for k in ("SSM_FORCE_LANES", "SSM_FORCE_CHUNKS", "SSM_FORCE_PATH")}

    def set_(**kw):
        for k, v in kw.items():
            key = "SSM_FORCE_" + k.upper()
            if v is None:
                os.environ.pop(key, None)
            else:
                os.environ[key] = str(v)
    yield set_
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def chunked(ssm, x, h0=None):
    return ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=h0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("lanes", [1, 2, 4])
@pytest.mark.parametrize("chunks", [1, 3])
def test_variants_with_carry(ssm, env, io, N, lanes, chunks):
    if lanes > N // 2:
        pytest.skip("variant needs at least two states per lane")
    env(lanes=lanes, chunks=chunks)
    # 70 channels: a partial block for every channels-per-CTA; L = 200 is a
    # multiple of 8 but not of the 16/32-step tile, so the last tile is ragged.
    x = I.make_scan_inputs(2, 70, N, 200, 1, io=io, recipe="scaled", seed=31, device="cuda", with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"io={io} N={N} lanes={lanes} chunks={chunks}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunks", [1, 2, 7])
def test_groups_partial_blocks(ssm, env, io, chunks):
    """G = 3 groups of 40 channels: each group's last channel block is partial,
    so the tile box overhangs the group edge; the next group's y and state must
    come out right (loads zero-fill, stores clip at the group edge)."""
    env(chunks=chunks)
    x = I.make_scan_inputs(2, 120, 16, 224, 3, io=io, recipe="scaled", seed=32, device="cuda", with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"groups chunks={chunks}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_single_pass_without_gate_skip_bias(ssm, io):
    x = I.make_scan_inputs(3, 64, 16, 96, 1, io=io, recipe="scaled", seed=33, device="cuda", with_z=False)
    y = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C)
    torch.cuda.synchronize()
    import oracle
    f = x.as_f64()
    assert_close(to_np(y), oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"]), io, "no z/D/bias")


def test_staged_matches_generic_path(ssm, env):
    x = I.make_scan_inputs(2, 96, 16, 256, 1, io="bf16", recipe="unit", seed=34, device="cuda")
    y_tma = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    env(path="generic")
    y_gen = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    ref = oracle_scan(x)
    assert_close(to_np(y_tma), ref, "bf16", "staged")
    assert_close(to_np(y_gen), ref, "bf16", "generic")
    # Both round the same fp32 readout to bf16; they may differ by one bf16 ulp
    # where the fp32 sums straddle a rounding boundary.
    diff = (y_tma.float() - y_gen.float()).abs()
    assert float((diff > 0).float().mean()) < 0.05


def test_staged_writes_only_y(ssm):
    x = I.make_scan_inputs(2, 20, 16, 96, 1, io="bf16", device="cuda", seed=35)
    n = x.u.numel()
    big = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = big[2048:2048 + n].view_as(x.u)
    ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, out=y)
    torch.cuda.synchronize()
    assert torch.all(big[:2048] == 7.0) and torch.all(big[2048 + n:] == 7.0)
    assert_close(to_np(y), oracle_scan(x), "bf16", "canary")


@pytest.mark.parametrize("chunks", [None, 1, 4, 16])
def test_bf16_b2_d1536_l2048_chunked_full(ssm, env, chunks):
    """bf16 I/O, fp32 state: batch 2, 1536 channels, N 16, L 2048 through the
    chunked entry point (the benchmark's launch configuration when chunks is
    None), whole tensor and final state against the oracle."""
    env(chunks=chunks)
    w = I.WORKLOADS["scan_bf16_b2_d1536_l2048"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16",
                           recipe=w["recipe"], seed=0, device="cuda")
    y, hf = chunked(ssm, x)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, final_state=True)
    e = assert_close(to_np(y), ref_y, "bf16", f"chunks={chunks}")
    eh = rel_l2(to_np(hf), ref_h)
    print(f"chunks={chunks}: y rel_l2 {e:.3e}, h_final rel_l2 {eh:.3e}")
    assert eh <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_summary_pass_with_other_lanes(ssm, env, io, monkeypatch):
    """The summary pass may share states over more lanes than the full pass.
    Its per-channel summaries do not depend on the split, so y and the final
    state must come out bit-identical to the one-lane summary pass; that run
    is checked against the oracle at the full tolerance.  The inputs are
    drawn on the CPU (then copied), so the same values can be evaluated
    without a GPU by the correctly rounded fp32 model of the CPU tests."""
    env(lanes=1, chunks=5)
    x = I.make_scan_inputs(2, 150, 16, 480, 1, io=io, recipe="scaled", seed=36, device="cpu",
                           with_h0=True).to("cuda")
    outs = {}
    for agg_lanes in (1, 2, 4):
        monkeypatch.setenv("SSM_FORCE_AGG_LANES", str(agg_lanes))
        outs[agg_lanes] = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    for agg_lanes in (2, 4):
        assert torch.equal(outs[agg_lanes][0], outs[1][0]), f"y differs with agg_lanes={agg_lanes}"
        assert torch.equal(outs[agg_lanes][1], outs[1][1]), f"h_final differs with agg_lanes={agg_lanes}"
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    y, hf = outs[1]
    assert_close(to_np(y), ref_y, io, "summary lanes")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_random_A(ssm, env, io):
    """A drawn per element (no pattern across states), time-chunked."""
    env(chunks=3)
    x = I.make_scan_inputs(2, 96, 16, 320, 1, io=io, recipe="scaled", seed=38, device="cuda", with_h0=True)
    x.A = I.a_values_random(96, 16, seed=38, device="cuda")
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, "random A")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
