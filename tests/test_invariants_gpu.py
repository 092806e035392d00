"""Structural invariants re-run on the GPU path: carried state across a
split, decode == scan, the vanishing-step limit, and the chunked entry point
against the oracle with an initial state."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_REL_L2, STATE_REL_L2, assert_close, oracle_compare_blocks, oracle_scan, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def chunked(ssm, x, h0=None, lo=0, hi=None):
    sl = slice(lo, hi)
    return ssm.scan_fwd_chunked(x.u[..., sl].contiguous(), x.delta[..., sl].contiguous(), x.A,
                                x.B[..., sl].contiguous(), x.C[..., sl].contiguous(),
                                z=None if x.z is None else x.z[..., sl].contiguous(), D=x.D,
                                dt_bias=x.dt_bias, h0=h0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunked_with_initial_state_matches_oracle(ssm, io):
    x = I.make_scan_inputs(2, 48, 16, 300, 2, io=io, recipe="scaled", seed=21, device="cuda",
                           with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, "chunked y")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2


@pytest.mark.parametrize("split", [1, 64, 100, 299])
def test_split_with_carried_state(ssm, split):
    x = I.make_scan_inputs(2, 40, 16, 300, 1, io="f32", recipe="scaled", seed=22, device="cuda",
                           with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    ya, ha = chunked(ssm, x, h0=x.h0, hi=split)
    yb, hb = chunked(ssm, x, h0=ha, lo=split)
    torch.cuda.synchronize()
    assert rel_l2(to_np(torch.cat([ya, yb], dim=2)), to_np(y)) <= 1e-6
    assert rel_l2(to_np(hb), to_np(hf)) <= 1e-6


def test_empty_sequence_returns_initial_state(ssm):
    x = I.make_scan_inputs(2, 16, 16, 0, 1, io="bf16", device="cuda", with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    assert torch.equal(hf, x.h0)
    _, hz = chunked(ssm, x, h0=None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hz) == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_steps_equal_scan(ssm, io):
    batch, dim, N, L = 3, 40, 16, 50
    x = I.make_scan_inputs(batch, dim, N, L, 1, io=io, recipe="scaled", seed=23, device="cuda",
                           with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    state = x.h0.clone()
    ys = []
    for t in range(L):
        ys.append(ssm.state_update(state, x.u[..., t].contiguous(), x.delta[..., t].contiguous(), x.A,
                                   x.B[..., t].contiguous(), x.C[..., t].contiguous(),
                                   z=x.z[..., t].contiguous(), D=x.D, dt_bias=x.dt_bias))
    torch.cuda.synchronize()
    yd = torch.stack(ys, dim=2)
    tol = 1e-5 if io == "f32" else 1e-2  # bf16: both outputs rounded independently
    assert rel_l2(to_np(yd), to_np(y)) <= tol
    assert rel_l2(to_np(state), to_np(hf)) <= 1e-5


def test_vanishing_step_leaves_skip_path(ssm):
    x = I.make_scan_inputs(2, 32, 16, 150, 1, io="f32", recipe="scaled", seed=24, device="cuda")
    x.dt_bias = torch.full_like(x.dt_bias, -60.0)
    y = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    f = x.as_f64()
    want = f["Dskip"][None, :, None] * f["u"] * (f["z"] / (1 + np.exp(-f["z"])))
    assert rel_l2(to_np(y), want) <= 1e-6


def test_long_sequence_final_state_full(ssm):
    """bf16 I/O, batch 1, 5120 channels, L 65536, final state returned, in the
    benchmark's launch configuration: every element of y and of h_final
    against the oracle (computed over blocks of channels)."""
    w = I.WORKLOADS["scan_bf16_b1_d5120_l65536_final_state"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16",
                           recipe=w["recipe"], seed=0, device="cuda")
    y, hf = chunked(ssm, x)
    torch.cuda.synchronize()
    e, eh, _ = oracle_compare_blocks(x, y, hf)
    print(f"b1 d5120 l65536: y rel_l2 {e:.3e}, h_final rel_l2 {eh:.3e}")
    assert e <= BF16_REL_L2, f"y rel_l2={e:.3e}"
    assert eh <= STATE_REL_L2, f"h_final rel_l2={eh:.3e}"
