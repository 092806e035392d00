"""Tensors past 2^31 elements on the GPU: every offset into them must be
64-bit.  The scan, the packed scan, the short convolution, the backward
pass and the SSD layer run on activations of more than 2^31 elements (bf16, 4.3 GB each) and the decode step on a state of 2^31 + 2^20
fp32 elements (8.6 GB); sampled channels -- at the start, in the middle and
at the end, whose elements lie beyond 2^31 -- are compared with the oracle
(for the backward pass, every per-channel gradient; dB and dC sum over all
channels and are checked on the smaller shapes of the backward tests).  The oracle
sees only the sampled rows (sliced on the device, then widened exactly), so
host memory stays small."""
import numpy as np
import pytest
import torch

import oracle
from parity import rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu

BF16_REL_L2 = 5e-3
STATE_REL_L2 = 1e-4


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def f64(t):
    return t.detach().to("cpu", torch.float32).double().numpy()


def test_scan_past_2_31_elements(ssm, monkeypatch):
    """The plan the library picks for this shape (one pass), then a forced
    split into four time chunks (summary, carry and fused passes)."""
    batch, dim, N, L = 1, 16400, 16, 131072
    assert batch * dim * L > 2 ** 31
    x = I.make_scan_inputs(batch, dim, N, L, 1, io="bf16", recipe="scaled", seed=41, device="cuda")
    channels = [0, dim // 2, dim - 17, dim - 1]
    assert (dim - 1) * L > 2 ** 31  # the last channel's first element
    B, C = f64(x.B), f64(x.C)
    A, D, bias = f64(x.A), f64(x.D), f64(x.dt_bias)
    refs = {}
    for d in channels:
        sl = slice(d, d + 1)
        refs[d] = oracle.scan(f64(x.u[:, sl]), f64(x.delta[:, sl]), A[sl], B, C, z=f64(x.z[:, sl]),
                              Dskip=D[sl], dt_bias=bias[sl], return_final_state=True)
    for chunks in (None, 4):
        if chunks is not None:
            monkeypatch.setenv("SSM_FORCE_CHUNKS", str(chunks))
            assert ssm.scan_plan(batch, dim, N, L, 1, torch.bfloat16)["chunks"] == chunks
        y, hf = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias)
        torch.cuda.synchronize()
        assert ssm.device_status() == 0
        for d in channels:
            sl = slice(d, d + 1)
            ry, rh = refs[d]
            e = rel_l2(f64(y[:, sl]), ry)
            eh = rel_l2(f64(hf[:, sl]), rh)
            assert e <= BF16_REL_L2, f"chunks={chunks} channel {d}: y rel_l2 {e:.3e}"
            assert eh <= STATE_REL_L2, f"chunks={chunks} channel {d}: h_final rel_l2 {eh:.3e}"
        del y, hf


def test_decode_step_past_2_31_state_elements(ssm):
    batch, dim, N = 2049, 65536, 16
    assert batch * dim * N > 2 ** 31
    state = I.make_decode_state(batch, dim, N, seed=43, device="cuda")
    tok = I.make_decode_token(batch, dim, N, step=0, io="bf16", recipe="scaled", seed=43, device="cuda")
    prm = I.decode_params(dim, N, recipe="scaled", seed=43, device="cuda")
    A, D, bias = prm["A"], prm["D"], prm["dt_bias"]
    rows = [(0, 0), (batch // 2, dim // 2), (batch - 1, dim - 3), (batch - 1, dim - 1)]
    before = {r: f64(state[r[0], r[1]]) for r in rows}
    y = ssm.state_update(state, tok["u"], tok["delta"], A, tok["B"], tok["C"], z=tok["z"], D=D, dt_bias=bias)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    An, Dn, bn = f64(A), f64(D), f64(bias)
    for b, d in rows:
        st = before[(b, d)].reshape(1, 1, N)
        rs, ry = oracle.state_update(st, f64(tok["u"][b:b + 1, d:d + 1]), f64(tok["delta"][b:b + 1, d:d + 1]),
                                     An[d:d + 1], f64(tok["B"][b:b + 1]), f64(tok["C"][b:b + 1]),
                                     z=f64(tok["z"][b:b + 1, d:d + 1]), Dskip=Dn[d:d + 1],
                                     dt_bias=bn[d:d + 1])
        es = rel_l2(f64(state[b, d]).reshape(1, 1, N), rs)
        assert es <= STATE_REL_L2, f"row {(b, d)}: state rel_l2 {es:.3e}"
        gy, ryv = float(f64(y[b, d])), float(ry[0, 0])
        assert abs(gy - ryv) <= 1e-2 * max(abs(ryv), 1e-2), f"row {(b, d)}: y {gy} against {ryv}"


def test_backward_past_2_31_elements(ssm):
    batch, dim, N, L = 1, 16400, 16, 131072
    x = I.make_scan_inputs(batch, dim, N, L, 1, io="bf16", recipe="scaled", seed=47, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(4700)
    dy = torch.randn((batch, dim, L), generator=g, device="cuda").to(torch.bfloat16)
    got = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    B, C = f64(x.B), f64(x.C)
    A, D, bias = f64(x.A), f64(x.D), f64(x.dt_bias)
    for d in [0, dim // 2, dim - 17, dim - 1]:
        sl = slice(d, d + 1)
        ref = oracle.scan_bwd(f64(x.u[:, sl]), f64(x.delta[:, sl]), A[sl], B, C, f64(dy[:, sl]),
                              z=f64(x.z[:, sl]), Dskip=D[sl], dt_bias=bias[sl])
        for k in ("du", "ddelta", "dz"):
            e = rel_l2(f64(got[k][:, sl]), ref[k])
            assert e <= BF16_REL_L2, f"channel {d}: {k} rel_l2 {e:.3e}"
        for k, tol in (("dA", 1e-3), ("dD", 1e-3), ("ddt_bias", 1e-3), ("dh0", 1e-3)):
            e = rel_l2(f64(got[k][sl] if got[k].dim() < 3 else got[k][:, sl]), ref[k])
            assert e <= tol, f"channel {d}: {k} rel_l2 {e:.3e}"


def test_ssd_past_2_31_elements(ssm):
    batch, nheads, P, N, L = 2, 64, 64, 128, 270336
    assert batch * nheads * P * L > 2 ** 31
    x = I.make_ssd_inputs(batch, nheads, P, N, L, 1, seed=49, device="cuda", with_h0=True)
    y, hf = ssm.ssd_fwd(x["x"], x["delta"], x["A"], x["B"], x["C"], z=x["z"], D=x["D"], dt_bias=x["dt_bias"],
                        h0=x["h0"], headdim=P, return_final_state=True)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    A, D, bias = f64(x["A"]), f64(x["D"]), f64(x["dt_bias"])
    for b, h in [(0, 0), (1, nheads // 2), (1, nheads - 1)]:
        ch = slice(h * P, (h + 1) * P)
        ry, rh = oracle.ssd(f64(x["x"][b:b + 1, ch]), f64(x["delta"][b:b + 1, h:h + 1]), A[h:h + 1],
                            f64(x["B"][b:b + 1]), f64(x["C"][b:b + 1]), z=f64(x["z"][b:b + 1, ch]),
                            Dskip=D[h:h + 1], dt_bias=bias[h:h + 1], h0=f64(x["h0"][b:b + 1, ch]),
                            headdim=P, return_final_state=True)
        e = rel_l2(f64(y[b:b + 1, ch]), ry)
        eh = rel_l2(f64(hf[b:b + 1, ch]), rh)
        assert e <= BF16_REL_L2, f"(b, h) = {(b, h)}: y rel_l2 {e:.3e}"
        assert eh <= STATE_REL_L2, f"(b, h) = {(b, h)}: h_final rel_l2 {eh:.3e}"


def _randn_cuda(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def test_conv1d_past_2_31_elements(ssm):
    batch, dim, L, W = 1, 16400, 131072, 4
    x = _randn_cuda((batch, dim, L), 51)
    w = _randn_cuda((dim, W), 52, torch.float32, W ** -0.5)
    bias = _randn_cuda((dim,), 53, torch.float32, 0.1)
    out = ssm.causal_conv1d(x, w, bias)
    torch.cuda.synchronize()
    for d in [0, dim // 2, dim - 17, dim - 1]:
        sl = slice(d, d + 1)
        ref = oracle.causal_conv1d(f64(x[:, sl]), f64(w[sl]), f64(bias[sl]))
        e = rel_l2(f64(out[:, sl]), ref)
        assert e <= BF16_REL_L2, f"channel {d}: rel_l2 {e:.3e}"


def test_packed_scan_past_2_31_elements(ssm):
    dim, N = 16384, 16
    lengths = [16385] * 8                     # T = 131080 steps: dim * T > 2^31
    T = sum(lengths)
    assert dim * T > 2 ** 31
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device="cuda")
    u, delta, z = (_randn_cuda((dim, T), s) for s in (61, 62, 63))
    B, C = (_randn_cuda((1, N, T), s, scale=N ** -0.5) for s in (64, 65))
    A = I.a_values(dim, N, "cuda")
    D = 1.0 + 0.1 * _randn_cuda((dim,), 66, torch.float32)
    bias = I.dt_bias_values(dim, 67, "cuda")
    y, hf = ssm.scan_fwd_varlen(u, delta, A, B, C, cu, z=z, D=D, dt_bias=bias, return_final_state=True)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    cun = cu.cpu().numpy()
    for d in [0, dim // 2, dim - 17, dim - 1]:
        sl = slice(d, d + 1)
        ry, rh = oracle.scan_varlen(f64(u[sl]), f64(delta[sl]), f64(A[sl]), f64(B), f64(C), cun,
                                    z=f64(z[sl]), Dskip=f64(D[sl]), dt_bias=f64(bias[sl]), return_final_state=True)
        e = rel_l2(f64(y[sl]), ry)
        eh = rel_l2(f64(hf[:, sl]), rh)
        assert e <= BF16_REL_L2, f"channel {d}: y rel_l2 {e:.3e}"
        assert eh <= STATE_REL_L2, f"channel {d}: h_final rel_l2 {eh:.3e}"
