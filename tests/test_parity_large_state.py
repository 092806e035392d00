"""GPU parity of the scan and decode step with large state sizes (N = 32, 64,
128 and 256, several lanes sharing one channel's states) against the fp64
oracle: the TMA-staged path single pass and time-chunked, the generic path,
the packed variable-length scan and the decode step.  N = 128 and 256 (8 or 16
lanes of 16 states) run on every path: on the generic one and in the packed
scan with the widened B/C tile in dynamic shared memory, single-buffered."""
import numpy as np
import pytest
import torch

import oracle
from parity import STATE_REL_L2, assert_close, oracle_scan, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def chunked(ssm, x, h0=None):
    return ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=h0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [32, 64, 128, 256])
@pytest.mark.parametrize("chunks", [1, 3])
def test_staged_large_state(ssm, monkeypatch, io, N, chunks):
    monkeypatch.setenv("SSM_FORCE_CHUNKS", str(chunks))
    # 70 channels (partial channel blocks), L = 200 (ragged last tile), 2 groups.
    x = I.make_scan_inputs(2, 70 * 2, N, 200, 2, io=io, recipe="scaled", seed=80 + N, device="cuda", with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"staged N={N} chunks={chunks} io={io}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N,lanes", [(32, 2), (32, 4), (32, 8), (64, 4), (64, 8), (128, 8), (256, 16)])
def test_generic_large_state(ssm, monkeypatch, io, N, lanes):
    monkeypatch.setenv("SSM_FORCE_PATH", "generic")
    monkeypatch.setenv("SSM_FORCE_LANES", str(lanes))
    x = I.make_scan_inputs(2, 96, N, 203, 1, io=io, recipe="scaled", seed=90 + N + lanes, device="cuda")
    y = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    assert_close(to_np(y), oracle_scan(x), io, f"generic N={N} lanes={lanes} io={io}")
    assert ssm.device_status() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N,L", [(128, 203), (256, 131)])
def test_unaligned_rows_large_state(ssm, io, N, L):
    """Rows that are not whole 16-byte packets (no TMA description): N = 128
    and 256 on the generic kernel, with an initial and a final state."""
    x = I.make_scan_inputs(2, 48, N, L, 2, io=io, recipe="scaled", seed=70 + N, device="cuda", with_h0=True)
    y, hf = chunked(ssm, x, h0=x.h0)
    torch.cuda.synchronize()
    assert not ssm.scan_plan(2, 48, N, L, 2, x.u.dtype)["staged"]
    ref_y, ref_h = oracle_scan(x, h0=x.h0, final_state=True)
    assert_close(to_np(y), ref_y, io, f"unaligned N={N} L={L} io={io}")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [32, 64, 128, 256])
def test_varlen_large_state(ssm, io, N):
    x = I.make_varlen_inputs(64, N, [37, 0, 90, 8], io=io, seed=95 + N, device="cuda", with_h0=True)
    y, hf = ssm.scan_fwd_varlen(x["u"], x["delta"], x["A"], x["B"], x["C"], x["cu_seqlens"], z=x["z"], D=x["D"],
                                dt_bias=x["dt_bias"], h0=x["h0"], return_final_state=True)
    torch.cuda.synchronize()
    f = lambda t: to_np(t)
    ry, rh = oracle.scan_varlen(f(x["u"]), f(x["delta"]), f(x["A"]), f(x["B"]), f(x["C"]),
                                x["cu_seqlens"].cpu().numpy(), z=f(x["z"]), Dskip=f(x["D"]),
                                dt_bias=f(x["dt_bias"]), h0=f(x["h0"]), return_final_state=True)
    assert_close(to_np(y), ry, io, f"varlen N={N} io={io}")
    assert rel_l2(to_np(hf), rh) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [32, 64, 128, 256])
def test_decode_large_state(ssm, io, N):
    prm = I.decode_params(200, N, device="cuda")
    state = I.make_decode_state(5, 200, N, seed=3, device="cuda")
    st0 = to_np(state)
    tok = I.make_decode_token(5, 200, N, 0, io=io, seed=4, device="cuda")
    y = ssm.state_update(state, tok["u"], tok["delta"], prm["A"], tok["B"], tok["C"], z=tok["z"], D=prm["D"],
                         dt_bias=prm["dt_bias"])
    torch.cuda.synchronize()
    ref_st, ref_y = oracle.state_update(st0, to_np(tok["u"]), to_np(tok["delta"]), to_np(prm["A"]), to_np(tok["B"]),
                                        to_np(tok["C"]), z=to_np(tok["z"]), Dskip=to_np(prm["D"]),
                                        dt_bias=to_np(prm["dt_bias"]))
    assert_close(to_np(y), ref_y, io, f"decode N={N} io={io}")
    assert rel_l2(to_np(state), ref_st) <= STATE_REL_L2


def test_n64_full_size_bf16_b2_d1536_l2048(ssm):
    """The benchmark's N = 64 shape in full (its own launch plan), every output."""
    w = I.WORKLOADS["scan_bf16_b2_d1536_l2048_n64"]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16", recipe=w["recipe"],
                           seed=0, device="cuda")
    y, hf = chunked(ssm, x)
    torch.cuda.synchronize()
    ref_y, ref_h = oracle_scan(x, final_state=True)
    e = assert_close(to_np(y), ref_y, "bf16", "N=64 b2 d1536 L2048")
    assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    print(f"N=64 full-size rel_l2 = {e:.3e}")


def test_n128_single_pass_and_other_forms(ssm):
    """N = 128 through the entry point without a workspace (one pass), on a
    row that is not whole 16-byte packets (the generic kernel), and in the
    packed scan, each against the oracle."""
    x = I.make_scan_inputs(2, 48, 128, 96, 1, io="bf16", recipe="scaled", seed=7, device="cuda")
    y = ssm.scan_fwd(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    assert_close(to_np(y), oracle_scan(x), "bf16", "N=128 single pass")
    odd = I.make_scan_inputs(1, 16, 128, 37, 1, io="bf16", recipe="scaled", seed=8, device="cuda")
    yo = ssm.scan_fwd(odd.u, odd.delta, odd.A, odd.B, odd.C, z=odd.z, D=odd.D, dt_bias=odd.dt_bias)
    torch.cuda.synchronize()
    assert_close(to_np(yo), oracle_scan(odd), "bf16", "N=128 unaligned row")
    v = I.make_varlen_inputs(16, 128, [5, 11], io="bf16", seed=9, device="cuda", row_multiple=8)
    yv = ssm.scan_fwd_varlen(v["u"], v["delta"], v["A"], v["B"], v["C"], v["cu_seqlens"], z=v["z"], D=v["D"],
                             dt_bias=v["dt_bias"])
    torch.cuda.synchronize()
    f = lambda t: to_np(t)
    ry = oracle.scan_varlen(f(v["u"]), f(v["delta"]), f(v["A"]), f(v["B"]), f(v["C"]), v["cu_seqlens"].cpu().numpy(),
                            z=f(v["z"]), Dskip=f(v["D"]), dt_bias=f(v["dt_bias"]))
    n = int(v["cu_seqlens"][-1])  # the row's padding past the last sequence is not written
    assert_close(to_np(yv)[:, :n], ry[:, :n], "bf16", "N=128 packed")
    assert ssm.device_status() == 0
