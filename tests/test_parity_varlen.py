"""GPU parity of the packed variable-length scan and of the decode step on a
pool of state slots against the fp64 oracle: mixed lengths including empty
and one-token sequences, starts on and off the 16-byte packet boundary, two
groups, h0 and h_final, every lanes-per-channel variant; padding rows and
untouched slots of the pool."""
import numpy as np
import pytest
import torch

import oracle
from parity import STATE_REL_L2, assert_close, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def f64(t):
    return None if t is None else to_np(t)


def run_varlen(ssm, x, **kw):
    return ssm.scan_fwd_varlen(x["u"], x["delta"], x["A"], x["B"], x["C"], x["cu_seqlens"], z=x["z"], D=x["D"],
                               dt_bias=x["dt_bias"], h0=x.get("h0"), return_final_state=True, **kw)


def oracle_varlen(x):
    return oracle.scan_varlen(f64(x["u"]), f64(x["delta"]), f64(x["A"]), f64(x["B"]), f64(x["C"]),
                              x["cu_seqlens"].cpu().numpy(), z=f64(x["z"]), Dskip=f64(x["D"]),
                              dt_bias=f64(x["dt_bias"]), h0=f64(x.get("h0")), return_final_state=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("lanes", [1, 2, 4, 8])
def test_varlen_mixed_lengths(ssm, monkeypatch, io, lanes):
    monkeypatch.setenv("SSM_FORCE_LANES", str(lanes))
    lengths = [37, 0, 1, 200, 64, 5, 130]   # starts 0, 37, 37, 38, 238, 302, 307: most off the packet boundary
    x = I.make_varlen_inputs(96, 16, lengths, ngroups=2, io=io, seed=50 + lanes, device="cuda", with_h0=True)
    y, hf = run_varlen(ssm, x)
    torch.cuda.synchronize()
    ry, rh = oracle_varlen(x)
    assert_close(to_np(y), ry, io, f"varlen io={io} lanes={lanes}")
    assert rel_l2(to_np(hf), rh) <= STATE_REL_L2
    np.testing.assert_array_equal(to_np(hf[1]), to_np(x["h0"][1]))  # the empty sequence keeps its h0


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_varlen_padded_row(ssm, io):
    """Mixed lengths in a row padded to a multiple of 8 steps (whole-packet
    loads for every channel row); the padding's y is not compared."""
    lengths = [37, 0, 1, 200, 64, 5, 130]
    x = I.make_varlen_inputs(96, 16, lengths, ngroups=2, io=io, seed=58, device="cuda", with_h0=True,
                             row_multiple=8)
    y, hf = run_varlen(ssm, x)
    torch.cuda.synchronize()
    ry, rh = oracle_varlen(x)
    n = int(x["cu_seqlens"][-1])
    assert x["u"].shape[1] % 8 == 0 and x["u"].shape[1] > n
    assert_close(to_np(y)[:, :n], ry[:, :n], io, f"varlen padded row io={io}")
    assert rel_l2(to_np(hf), rh) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_varlen_aligned_lengths_without_h0(ssm, io):
    """Lengths that keep every start on the packet boundary (vector loads)."""
    lengths = [64, 128, 8, 256]
    x = I.make_varlen_inputs(130, 16, lengths, io=io, seed=60, device="cuda")
    y, hf = run_varlen(ssm, x)
    torch.cuda.synchronize()
    ry, rh = oracle_varlen(x)
    assert_close(to_np(y), ry, io, f"varlen aligned io={io}")
    assert rel_l2(to_np(hf), rh) <= STATE_REL_L2


def test_varlen_one_sequence_matches_the_scan(ssm):
    x = I.make_varlen_inputs(64, 16, [300], io="bf16", seed=61, device="cuda", with_h0=True)
    y, hf = run_varlen(ssm, x)
    y2, hf2 = ssm.scan_fwd_chunked(x["u"][None], x["delta"][None], x["A"], x["B"][None], x["C"][None],
                                   z=x["z"][None], D=x["D"], dt_bias=x["dt_bias"], h0=x["h0"])
    torch.cuda.synchronize()
    ry, rh = oracle_varlen(x)
    assert_close(to_np(y), ry, "bf16", "varlen one sequence")
    assert_close(to_np(y2[0]), ry, "bf16", "chunked scan")
    assert rel_l2(to_np(hf2), rh) <= STATE_REL_L2


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["staged", "generic"])
def test_pooled_decode(ssm, monkeypatch, io, path):
    if path == "generic":
        monkeypatch.setenv("SSM_FORCE_PATH", "generic")
    slots, batch, dim, N = 9, 6, 256, 16
    pool = I.make_decode_state(slots, dim, N, seed=70, device="cuda")
    idx = torch.tensor([4, -1, 0, 8, 99, 2], dtype=torch.int32, device="cuda")   # -1 and 99: padding rows
    prm = I.decode_params(dim, N, device="cuda")
    tok = I.make_decode_token(batch, dim, N, 0, io=io, seed=71, device="cuda")
    pool0 = pool.clone()
    y = torch.full((batch, dim), 7.0, dtype=tok["u"].dtype, device="cuda")
    ssm.state_update(pool, tok["u"], tok["delta"], prm["A"], tok["B"], tok["C"], z=tok["z"], D=prm["D"],
                     dt_bias=prm["dt_bias"], out=y, state_indices=idx)
    torch.cuda.synchronize()
    ref_idx = np.array([4, -1, 0, 8, -1, 2], dtype=np.int32)
    ref_pool, ry = oracle.state_update_indexed(f64(pool0), ref_idx, f64(tok["u"]), f64(tok["delta"]), f64(prm["A"]),
                                               f64(tok["B"]), f64(tok["C"]), z=f64(tok["z"]), Dskip=f64(prm["D"]),
                                               dt_bias=f64(prm["dt_bias"]))
    live = ref_idx >= 0
    got = to_np(y)
    assert_close(got[live], ry[live], io, f"pooled decode {path}")
    assert np.all(got[~live] == 7.0), "padding rows must not be written"
    assert rel_l2(to_np(pool), ref_pool) <= STATE_REL_L2
    untouched = [s for s in range(slots) if s not in (4, 0, 8, 2)]
    assert torch.equal(pool[untouched], pool0[untouched])
    assert ssm.device_status() == 0
