"""The launch plan (host-only, no GPU): the staged kernels' lanes and time
chunks for the benchmark's workloads are the ones measured best on B300 (or
within a few percent of it), and the plan follows the argument rules."""
import pytest
import torch

from selective_state_space_109_b300 import build


@pytest.fixture(scope="module")
def ssm():
    build.build()
    from selective_state_space_109_b300 import ssm as m
    return m


@pytest.mark.parametrize("shape,lanes,chunks", [
    ((2, 1536, 16, 2048), 2, 12),
    ((8, 2048, 16, 4096), 2, 1),
    ((1, 5120, 16, 65536), 1, 59),    # the headline call: 2182 us against 2225 us at 29 chunks
    ((2, 1536, 32, 2048), 2, 12),
    ((2, 1536, 64, 2048), 4, 6),
    ((2, 1536, 128, 2048), 8, 1),
    ((2, 1536, 256, 2048), 16, 3),    # 872 us against 938 us in one pass
])
def test_plans_of_the_measured_workloads(ssm, shape, lanes, chunks):
    b, d, n, L = shape
    plan = ssm.scan_plan(b, d, n, L, 1, torch.bfloat16)
    assert plan["staged"] and plan["lanes"] == lanes and plan["chunks"] == chunks
    assert plan["kernels"] == (3 if chunks > 1 else 1)


def test_plan_rules(ssm):
    # a state split over lanes keeps at most 16 states a lane
    for n in (4, 8, 16, 32, 64, 128, 256):
        p = ssm.scan_plan(4, 512, n, 4096, 1, torch.bfloat16)
        assert n // p["lanes"] <= 16 and n // p["lanes"] >= 2
    # without a workspace the call never splits time
    assert ssm.scan_plan(2, 1536, 16, 2048, 1, torch.bfloat16, chunked=False)["chunks"] == 1
    # rows that are not whole 16-byte packets take the generic kernel
    assert not ssm.scan_plan(2, 64, 16, 2047, 1, torch.bfloat16)["staged"]
    # the chunk count never exceeds 64 nor the tiles of the sequence
    assert ssm.scan_plan(1, 16, 16, 64, 1, torch.bfloat16)["chunks"] <= 4
    assert ssm.scan_plan(1, 64, 16, 1 << 20, 1, torch.float32)["chunks"] <= 64
    # N = 128 on rows that are not whole 16-byte packets: the register-staged kernel
    p128 = ssm.scan_plan(1, 64, 128, 2047, 1, torch.bfloat16)
    assert not p128["staged"] and p128["chunks"] == 1 and p128["kernels"] == 1
