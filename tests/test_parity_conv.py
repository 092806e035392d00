"""GPU parity of the short causal convolution in front of the scan (and its
decode step) against the fp64 oracle: widths 1-4, fp32 and bf16 I/O, with
and without bias, history in and out, rows whose byte length is a multiple of
16 (vector path, including lengths that leave a warp spanning two rows) and
ragged ones (element path)."""
import numpy as np
import pytest
import torch

import oracle
from parity import F32_MAX_REL, F32_REL_L2, max_rel, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def make(batch, dim, L, W, io, seed, bias=True, history=True):
    c = I.make_conv_inputs(batch, dim, L, W, io=io, seed=seed, device="cuda", with_prev=history)
    return c["x"], c["w"], c["bias"] if bias else None, c["x_prev"]


def f64(t):
    return None if t is None else to_np(t)


def check(got, ref, io, what):
    e2 = rel_l2(got, ref)
    if io == "f32":
        em = max_rel(got, ref)
        assert e2 <= F32_REL_L2 and em <= F32_MAX_REL, f"{what}: rel_l2={e2:.2e} max_rel={em:.2e}"
    else:
        # bf16 output: one rounding of the fp32 result (relative 2^-8), so the
        # error of every element is bounded by its own magnitude.
        err = np.abs(got - ref)
        assert np.all(err <= (2.0 ** -8 + 2e-6) * np.abs(ref) + 1e-6), f"{what}: max err {err.max():.3e}"
        assert e2 <= 5e-3, f"{what}: rel_l2={e2:.2e}"


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [8, 200, 203, 1024])
def test_conv_forward(ssm, io, W, L):
    x, w, b, prev = make(3, 37, L, W, io, seed=W * 1000 + L)
    last = torch.empty_like(prev) if prev is not None and W > 1 else None
    out = ssm.causal_conv1d(x, w, b, prev if W > 1 else None, x_last=last)
    torch.cuda.synchronize()
    ref, ref_last = oracle.causal_conv1d(f64(x), f64(w), f64(b), f64(prev) if W > 1 else None, return_last=True)
    check(to_np(out), ref, io, f"io={io} W={W} L={L}")
    if last is not None:
        np.testing.assert_array_equal(to_np(last), ref_last)
    assert ssm.device_status() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_without_bias_history_or_silu(ssm, io):
    x, w, _, _ = make(2, 64, 96, 4, io, seed=5, bias=False, history=False)
    out = ssm.causal_conv1d(x, w, silu=False)
    torch.cuda.synchronize()
    check(to_np(out), oracle.causal_conv1d(f64(x), f64(w), silu=False), io, "plain conv")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_segments_chain(ssm, io):
    """Three segments, each taking the previous one's history: equal to one pass."""
    x, w, b, prev = make(2, 48, 3 * 64, 4, io, seed=9)
    ref = oracle.causal_conv1d(f64(x), f64(w), f64(b), f64(prev))
    h = [prev.clone(), torch.empty_like(prev)]
    outs = []
    for s in range(3):
        outs.append(ssm.causal_conv1d(x[:, :, 64 * s:64 * (s + 1)].contiguous(), w, b, h[s % 2], x_last=h[(s + 1) % 2]))
    torch.cuda.synchronize()
    check(np.concatenate([to_np(o) for o in outs], axis=2), ref, io, "segments")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 4])
def test_conv_decode_steps(ssm, io, W):
    x, w, b, prev = make(4, 40, 12, W, io, seed=13 + W)
    state = prev.clone() if W > 1 else None
    ref_state = f64(prev) if W > 1 else np.zeros((4, 40, 0))
    for t in range(12):
        out = ssm.causal_conv1d_update(state, x[:, :, t].contiguous(), w, b)
        torch.cuda.synchronize()
        ref_state, ref = oracle.causal_conv1d_update(ref_state, f64(x[:, :, t]), f64(w), f64(b))
        check(to_np(out), ref, io, f"decode step {t}")
        if W > 1:
            np.testing.assert_array_equal(to_np(state), ref_state)


def test_conv_headline_shape_sampled(ssm):
    """bf16, batch 2 x 1536 channels x L 2048, W 4 (the scan workload's u):
    whole-tensor comparison against the oracle."""
    x, w, b, prev = make(2, 1536, 2048, 4, "bf16", seed=0, history=False)
    out = ssm.causal_conv1d(x, w, b)
    torch.cuda.synchronize()
    check(to_np(out), oracle.causal_conv1d(f64(x), f64(w), f64(b)), "bf16", "b2 d1536 L2048")
