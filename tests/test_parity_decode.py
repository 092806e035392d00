"""GPU decode state update vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_REL_L2, STATE_REL_L2, assert_close, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def run_step(ssm, state, tok, prm, **kw):
    return ssm.state_update(state, tok["u"], tok["delta"], prm["A"], tok["B"], tok["C"],
                            z=tok["z"], D=prm["D"], dt_bias=prm["dt_bias"], **kw)


@pytest.fixture
def path(request, monkeypatch):
    if request.param == "generic":
        monkeypatch.setenv("SSM_FORCE_PATH", "generic")
    elif request.param == "tma":  # the CTA-synchronous bulk-staged kernel
        monkeypatch.setenv("SSM_DECODE_KERNEL", "tma")
    return request.param


@pytest.mark.parametrize("path", [None, "tma", "generic"], indirect=True)
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("G", [1, 2])
def test_small_steps_whole_tensor(ssm, io, N, G, path):
    """The three decode kernels: bulk-staged warp-specialised (default),
    bulk-staged CTA-synchronous, and register-staged."""
    batch, dim = 11, 70  # 70 channels: a partial channel block; 11 sequences: a partial batch chunk
    prm = I.decode_params(dim, N, recipe="scaled", seed=1, device="cuda")
    state = I.make_decode_state(batch, dim, N, seed=1, device="cuda")
    ref_state = to_np(state)
    f = {k: to_np(v) for k, v in prm.items()}
    for step in range(5):
        tok = I.make_decode_token(batch, dim, N, step, ngroups=G, io=io, seed=1, device="cuda")
        y = run_step(ssm, state, tok, prm)
        torch.cuda.synchronize()
        t = {k: to_np(v) for k, v in tok.items()}
        ref_state, ref_y = oracle.state_update(ref_state, t["u"], t["delta"], f["A"], t["B"], t["C"],
                                               z=t["z"], Dskip=f["D"], dt_bias=f["dt_bias"])
        assert_close(to_np(y), ref_y, io, f"step {step}")
        assert rel_l2(to_np(state), ref_state) <= STATE_REL_L2


def test_decode_b256_d5120_1024_steps_sampled(ssm):
    """Full-size decode (batch 256, 5120 channels, N 16, fp32 state resident in
    HBM, one bf16 token per call) for 1024 consecutive steps; 24 x 40 sampled
    (sequence, channel) rows follow the oracle at every step."""
    w = I.WORKLOADS["decode_b256_d5120"]
    batch, dim, N = w["batch"], w["dim"], w["dstate"]
    prm = I.decode_params(dim, N, recipe="scaled", seed=0, device="cuda")
    state = I.make_decode_state(batch, dim, N, seed=0, device="cuda")
    rng = np.random.default_rng(0)
    bs = np.sort(rng.choice(batch, 24, replace=False))
    ds = np.sort(rng.choice(dim, 40, replace=False))
    bs_t = torch.as_tensor(bs, device="cuda")
    ds_t = torch.as_tensor(ds, device="cuda")
    ref_state = to_np(state[bs_t][:, ds_t])
    f = {k: to_np(v) for k, v in prm.items()}
    fA, fD, fb = f["A"][ds], f["D"][ds], f["dt_bias"][ds]
    worst = 0.0
    for step in range(w["steps"]):
        tok = I.make_decode_token(batch, dim, N, step, io="bf16", seed=0, device="cuda")
        y = run_step(ssm, state, tok, prm)
        sub = {k: to_np(v[bs_t][:, ds_t]) if k in ("u", "delta", "z") else to_np(v[bs_t])
               for k, v in tok.items()}
        ref_state, ref_y = oracle.state_update(ref_state, sub["u"], sub["delta"], fA, sub["B"],
                                               sub["C"], z=sub["z"], Dskip=fD, dt_bias=fb)
        e = rel_l2(to_np(y[bs_t][:, ds_t]), ref_y)
        worst = max(worst, e)
        assert e <= BF16_REL_L2, f"step {step}: rel_l2 {e:.3e}"
    es = rel_l2(to_np(state[bs_t][:, ds_t]), ref_state)
    print(f"worst per-step y rel_l2 {worst:.3e}; state rel_l2 after {w['steps']} steps {es:.3e}")
    assert es <= STATE_REL_L2


def test_decode_b256_d5120_full_tensor_steps(ssm):
    """Full-size decode (batch 256, 5120 channels, N 16), the launch the
    benchmark times: three consecutive steps on one resident state, every
    element of y and of the state against the oracle."""
    w = I.WORKLOADS["decode_b256_d5120"]
    batch, dim, N = w["batch"], w["dim"], w["dstate"]
    prm = I.decode_params(dim, N, recipe="scaled", seed=0, device="cuda")
    state = I.make_decode_state(batch, dim, N, seed=0, device="cuda")
    ref_state = to_np(state)
    f = {k: to_np(v) for k, v in prm.items()}
    for step in range(3):
        tok = I.make_decode_token(batch, dim, N, step, io="bf16", seed=0, device="cuda")
        y = run_step(ssm, state, tok, prm)
        torch.cuda.synchronize()
        t = {k: to_np(v) for k, v in tok.items()}
        ref_state, ref_y = oracle.state_update(ref_state, t["u"], t["delta"], f["A"], t["B"], t["C"],
                                               z=t["z"], Dskip=f["D"], dt_bias=f["dt_bias"])
        e = rel_l2(to_np(y), ref_y)
        es = rel_l2(to_np(state), ref_state)
        print(f"step {step}: y rel_l2 {e:.3e}, state rel_l2 {es:.3e}")
        assert e <= BF16_REL_L2, f"step {step}: y rel_l2 {e:.3e}"
        assert es <= STATE_REL_L2, f"step {step}: state rel_l2 {es:.3e}"


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dim,G", [(200, 1), (512, 2), (384, 1)])
def test_staged_decode_steps(ssm, io, dim, G):
    """Shapes the TMA-staged decode takes (N 16, 16-byte token rows, 128-channel
    blocks inside a group): a ragged last block (200), two groups (512), and
    full blocks (384); several consecutive steps on one state."""
    batch, N = 13, 16
    prm = I.decode_params(dim, N, recipe="scaled", seed=3, device="cuda")
    state = I.make_decode_state(batch, dim, N, seed=3, device="cuda")
    ref_state = to_np(state)
    f = {k: to_np(v) for k, v in prm.items()}
    for step in range(4):
        tok = I.make_decode_token(batch, dim, N, step, ngroups=G, io=io, seed=3, device="cuda")
        y = run_step(ssm, state, tok, prm)
        torch.cuda.synchronize()
        t = {k: to_np(v) for k, v in tok.items()}
        ref_state, ref_y = oracle.state_update(ref_state, t["u"], t["delta"], f["A"], t["B"], t["C"],
                                               z=t["z"], Dskip=f["D"], dt_bias=f["dt_bias"])
        assert_close(to_np(y), ref_y, io, f"step {step}")
        assert rel_l2(to_np(state), ref_state) <= STATE_REL_L2
    assert ssm.device_status() == 0


@pytest.mark.parametrize("path", [None, "tma"], indirect=True)
def test_decode_writes_exactly_its_state_and_y(ssm, path):
    """Canary: the state and y are views into larger buffers filled with a
    sentinel; 200 channels (a partial 128-channel block, and a partial 32-row
    box for the warp-specialised kernel's per-warp state stores), 3 steps."""
    batch, dim, N = 5, 200, 16
    prm = I.decode_params(dim, N, recipe="scaled", seed=2, device="cuda")
    s0 = I.make_decode_state(batch, dim, N, seed=2, device="cuda")
    n = s0.numel()
    big = torch.full((n + 8192,), 7.0, dtype=torch.float32, device="cuda")
    state = big[4096:4096 + n].view_as(s0)
    state.copy_(s0)
    ref_state = to_np(s0)
    f = {k: to_np(v) for k, v in prm.items()}
    big_y = torch.full((batch * dim + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = big_y[2048:2048 + batch * dim].view(batch, dim)
    for step in range(3):
        tok = I.make_decode_token(batch, dim, N, step, io="bf16", seed=2, device="cuda")
        run_step(ssm, state, tok, prm, out=y)
        torch.cuda.synchronize()
        t = {k: to_np(v) for k, v in tok.items()}
        ref_state, ref_y = oracle.state_update(ref_state, t["u"], t["delta"], f["A"], t["B"], t["C"],
                                               z=t["z"], Dskip=f["D"], dt_bias=f["dt_bias"])
        assert_close(to_np(y), ref_y, "bf16", f"step {step}")
        assert rel_l2(to_np(state), ref_state) <= STATE_REL_L2
    assert torch.all(big[:4096] == 7.0) and torch.all(big[4096 + n:] == 7.0)
    assert torch.all(big_y[:2048] == 7.0) and torch.all(big_y[2048 + batch * dim:] == 7.0)
