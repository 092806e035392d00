"""GPU forward scan vs the fp64 oracle on identical seeded inputs.

Small cases run the whole tensor through the oracle and span several tiles,
ragged tails, partial channel blocks, groups and every lanes-per-channel
variant; the two large workloads run at full size on the GPU, in the launch
configuration the benchmark times, and are compared element by element with
the oracle run over blocks of channels."""
import os

import numpy as np
import pytest
import torch

from parity import (BF16_REL_L2, STATE_REL_L2, assert_close, oracle_compare_blocks, oracle_scan, rel_l2,
                    to_np)
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


@pytest.fixture
def force_lanes():
    old = os.environ.get("SSM_FORCE_LANES")

    def set_(v):
        if v is None:
            os.environ.pop("SSM_FORCE_LANES", None)
        else:
            os.environ["SSM_FORCE_LANES"] = str(v)
    yield set_
    set_(old)


def run(ssm, x, **kw):
    return ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, **kw)


def test_tiny_f32_workload(ssm):
    """fp32 I/O, batch 1, 64 channels, N 16, L 256, G 1 (seed 0)."""
    w = I.WORKLOADS["scan_f32_tiny"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"],
                           io="f32", recipe="unit", seed=0, device="cuda")
    y = run(ssm, x)
    torch.cuda.synchronize()
    assert_close(to_np(y), oracle_scan(x), "f32", "tiny f32")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("lanes", [1, 2, 4, 8])
def test_every_variant_small(ssm, force_lanes, io, N, lanes):
    if lanes > N // 2:
        pytest.skip("variant needs at least two states per lane")
    force_lanes(lanes)
    # L = 203: several 64-step tiles plus a ragged tail, not a multiple of any packet.
    x = I.make_scan_inputs(2, 37, N, 203, 1, io=io, recipe="unit", seed=11, device="cuda")
    y = run(ssm, x)
    torch.cuda.synchronize()
    assert_close(to_np(y), oracle_scan(x), io, f"io={io} N={N} lanes={lanes}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 2, 7, 8, 63, 64, 65, 128, 200, 256, 1000])
def test_lengths(ssm, io, L):
    x = I.make_scan_inputs(1, 24, 16, L, 1, io=io, recipe="unit", seed=L, device="cuda")
    y = run(ssm, x)
    torch.cuda.synchronize()
    assert_close(to_np(y), oracle_scan(x), io, f"L={L}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_groups_and_optional_tensors(ssm, force_lanes, io):
    for lanes in (1, 4):
        force_lanes(lanes)
        x = I.make_scan_inputs(3, 96, 16, 130, 4, io=io, recipe="scaled", seed=5, device="cuda")
        y = run(ssm, x)
        torch.cuda.synchronize()
        assert_close(to_np(y), oracle_scan(x), io, f"groups lanes={lanes}")
        # no gate, no skip, no bias
        x2 = I.make_scan_inputs(3, 96, 16, 130, 4, io=io, recipe="scaled", seed=6, device="cuda",
                                with_z=False)
        x2.D = None
        x2.dt_bias = None
        y2 = ssm.scan_fwd(x2.u, x2.delta, x2.A, x2.B, x2.C)
        torch.cuda.synchronize()
        f = x2.as_f64()
        import oracle
        ref = oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"])
        assert_close(to_np(y2), ref, io, f"no z/D/bias lanes={lanes}")


def test_empty_sequence_and_batch(ssm):
    x = I.make_scan_inputs(2, 8, 16, 0, 1, io="bf16", device="cuda")
    y = run(ssm, x)
    assert y.shape == (2, 8, 0)
    x = I.make_scan_inputs(0, 8, 16, 16, 1, io="bf16", device="cuda")
    y = run(ssm, x)
    assert y.shape == (0, 8, 16)


def test_output_does_not_spill_past_its_rows(ssm):
    """Canary: y is a view into a larger buffer filled with a sentinel; the
    kernel must write exactly the y elements."""
    x = I.make_scan_inputs(2, 20, 16, 77, 1, io="bf16", device="cuda", seed=9)
    n = x.u.numel()
    big = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = big[2048:2048 + n].view_as(x.u)
    run(ssm, x, out=y)
    torch.cuda.synchronize()
    assert torch.all(big[:2048] == 7.0) and torch.all(big[2048 + n:] == 7.0)
    assert_close(to_np(y), oracle_scan(x), "bf16", "canary")


def test_bf16_b2_d1536_l2048_full(ssm):
    """bf16 I/O, fp32 state: batch 2, 1536 channels, N 16, L 2048; whole tensor."""
    w = I.WORKLOADS["scan_bf16_b2_d1536_l2048"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16",
                           recipe=w["recipe"], seed=0, device="cuda")
    y = run(ssm, x)
    torch.cuda.synchronize()
    e = assert_close(to_np(y), oracle_scan(x), "bf16", "b2 d1536 l2048")
    print(f"rel_l2 = {e:.3e}")


def test_bf16_b8_d2048_l4096_full(ssm):
    """bf16 I/O: batch 8, 2048 channels, L 4096 at full size; every element of
    y against the oracle (computed over blocks of channels)."""
    w = I.WORKLOADS["scan_bf16_b8_d2048_l4096"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16",
                           recipe=w["recipe"], seed=0, device="cuda")
    y = run(ssm, x)
    torch.cuda.synchronize()
    e, _, _ = oracle_compare_blocks(x, y)
    print(f"b8 d2048 l4096: y rel_l2 {e:.3e} over {y.numel()} elements")
    assert e <= BF16_REL_L2, f"rel_l2={e:.3e}"
