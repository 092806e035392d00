"""GPU parity of the backward pass (ssm_scan_bwd) against the fp64 oracle's
backward, on the same seeded inputs (bf16 inputs are widened exactly).

Sizes span several time chunks (128 to 160 steps, 64 at N = 64) with a ragged last
tile, channel blocks that end inside a group, two groups, and every optional
input present or absent; the benchmark's b2 d1536 N16 L2048 bf16 shape is
compared in full.

Tolerances.  Per-element outputs (du, ddelta, dz) follow the forward pass:
rel-L2 1e-5 for fp32 I/O, 5e-3 for bf16 I/O (outputs rounded to bf16).  The
fp32 sums (dA, dB, dC, dD, ddt_bias) and dh0 are reductions of O(L) to
O(batch * dim * L) products accumulated in fp32 in an order set by the
atomics: rel-L2 1e-4 for fp32 I/O, and 1e-3 for bf16 I/O, where the kernels
use MUFU exp/log (relative error ~1e-6 per step, compounded along the
recurrence)."""
import numpy as np
import pytest
import torch

import oracle
from parity import rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu

ELEM = ("du", "ddelta", "dz")
SUMS = ("dA", "dB", "dC", "dD", "ddt_bias", "dh0")
TOL = {"f32": (1e-5, 1e-4), "bf16": (5e-3, 1e-3)}


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def run_case(ssm, batch, dim, N, L, G, io, seed, gated=True, with_D=True, with_bias=True, with_h0=True,
             with_dhf=True, recipe="scaled"):
    x = I.make_scan_inputs(batch, dim, N, L, G, io=io, recipe=recipe, seed=seed, device="cuda", with_z=gated,
                           with_h0=with_h0)
    dt = x.u.dtype
    g = torch.Generator(device="cpu").manual_seed(1000 + seed)
    dy = torch.randn((batch, dim, L), generator=g).to(dt).cuda()
    dhf = torch.randn((batch, dim, N), generator=g).cuda() if with_dhf else None
    D = x.D if with_D else None
    bias = x.dt_bias if with_bias else None
    got = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=D, dt_bias=bias, h0=x.h0, dh_final=dhf)
    torch.cuda.synchronize()
    f = x.as_f64()
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], to_np(dy), z=f["z"],
                          Dskip=f["Dskip"] if with_D else None, dt_bias=f["dt_bias"] if with_bias else None,
                          h0=f["h0"], dh_final=None if dhf is None else to_np(dhf))
    return got, ref


def check(got, ref, io, what):
    te, ts = TOL[io]
    errs = {}
    for k in ELEM + SUMS:
        if got.get(k) is None:
            continue
        e = rel_l2(to_np(got[k]), ref[k])
        errs[k] = e
        assert np.all(np.isfinite(to_np(got[k]))), f"{what}: {k} has non-finite values"
        assert e <= (te if k in ELEM else ts), f"{what}: {k} rel_l2={e:.3e} (all: {errs})"
    return errs


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 8, 16, 32, 64, 128, 256])
def test_bwd_matches_oracle(ssm, io, N):
    # 2 groups of 35 channels (channel blocks end inside a group); L = 300:
    # several chunks and a ragged last tile.
    got, ref = run_case(ssm, 2, 70, N, 300, 2, io, seed=N)
    check(got, ref, io, f"N={N} io={io}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(gated=False), dict(with_D=False, with_bias=False),
                                  dict(with_h0=False, with_dhf=False)])
def test_bwd_optional_inputs(ssm, io, opts):
    got, ref = run_case(ssm, 1, 64, 16, 200, 1, io, seed=7, **opts)
    check(got, ref, io, f"{opts} io={io}")
    if not opts.get("gated", True):
        assert got["dz"] is None


@pytest.mark.parametrize("L", [1, 7, 128, 129, 257])
def test_bwd_lengths(ssm, L):
    """One step, a partial tile, exactly one chunk, one step past it, and an
    odd length (element-wise row access, fp32 and bf16)."""
    for io in ("f32", "bf16"):
        got, ref = run_case(ssm, 2, 40, 16, L, 1, io, seed=L)
        check(got, ref, io, f"L={L} io={io}")


@pytest.mark.parametrize("N", [128, 256])
def test_bwd_odd_length_large_state(ssm, N):
    """An odd length at the large state sizes: scalar dB/dC adds, a ragged
    last tile (its padded steps must add nothing to the dB/dC staging that
    later tiles reuse), several chunks of 64 steps."""
    for io in ("f32", "bf16"):
        got, ref = run_case(ssm, 1, 40, N, 203, 1, io, seed=N + 203)
        check(got, ref, io, f"N={N} L=203 io={io}")


def test_bwd_empty_sequence(ssm):
    x = I.make_scan_inputs(2, 16, 16, 0, 1, io="f32", seed=3, device="cuda", with_h0=True)
    dhf = torch.randn((2, 16, 16), device="cuda")
    dy = torch.empty((2, 16, 0), device="cuda")
    got = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0, dh_final=dhf)
    torch.cuda.synchronize()
    assert torch.equal(got["dh0"], dhf)
    assert not got["dA"].any() and not got["dD"].any() and not got["ddt_bias"].any()


def test_bwd_full_size_bf16_b2_d1536_l2048(ssm):
    """The benchmark's shape in full (every gradient, every element)."""
    w = I.WORKLOADS["scan_bf16_b2_d1536_l2048"]
    got, ref = run_case(ssm, w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], "bf16", seed=11,
                        with_h0=False, with_dhf=False, recipe=w["recipe"])
    errs = check(got, ref, "bf16", "b2 d1536 L2048")
    print("full-size bwd rel_l2:", {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_chunk_length_between_the_defaults(ssm, io):
    """The chunk length is chosen per shape to fill whole waves of the main
    pass: b2 d1440 N16 L520 takes 17 tiles of 8 steps (four chunks of 136,
    136, 136 and 112 steps), a length the other cases never meet."""
    need = ssm.bwd_workspace_size(2, 1440, 16, 520, 1, torch.bfloat16 if io == "bf16" else torch.float32)
    assert need == 4 * 2 * 1440 * 16 * 3 * 4
    got, ref = run_case(ssm, 2, 1440, 16, 520, 1, io, seed=23)
    errs = check(got, ref, io, f"b2 d1440 L520 {io}")
    print("chunk-length case rel_l2:", {k: f"{v:.2e}" for k, v in errs.items()})


def test_bwd_matches_finite_difference_of_the_kernel(ssm):
    """Self-consistency on the GPU alone (fp32): the directional derivative
    of sum(y * dy) along a random direction, by central differences of the
    forward kernel, equals the gradients' inner product with that direction."""
    x = I.make_scan_inputs(1, 32, 16, 256, 1, io="f32", recipe="scaled", seed=5, device="cuda", with_h0=True)
    g = torch.Generator(device="cpu").manual_seed(5)
    dy = torch.randn((1, 32, 256), generator=g).cuda()
    gr = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0)
    names = ["u", "delta", "z", "A", "B", "C", "D", "dt_bias", "h0"]
    keys = ["du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddt_bias", "dh0"]
    base = {n: getattr(x, n).clone() for n in names}
    dirs = {n: torch.randn(base[n].shape, generator=g).cuda() for n in names}

    def loss(eps):
        a = {n: base[n] + eps * dirs[n] for n in names}
        y, _ = ssm.scan_fwd_chunked(a["u"], a["delta"], a["A"], a["B"], a["C"], z=a["z"], D=a["D"],
                                    dt_bias=a["dt_bias"], h0=a["h0"])
        return float((y.double() * dy.double()).sum())
    eps = 1e-3
    fd = (loss(eps) - loss(-eps)) / (2 * eps)
    an = sum(float((gr[k].double() * dirs[n].double()).sum()) for n, k in zip(names, keys))
    assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (fd, an)


def channel_slice_bwd(x, dy, d):
    """The oracle's backward for channel d over every batch row (B, C shared by
    the single group): per-channel outputs and the channel's dA, dD, ddt_bias.
    Only the channel's rows are copied to the host."""
    sl = lambda t: None if t is None else to_np(t[:, d:d + 1])
    return oracle.scan_bwd(sl(x.u), sl(x.delta), to_np(x.A[d:d + 1]), to_np(x.B), to_np(x.C), sl(dy), z=sl(x.z),
                           Dskip=to_np(x.D[d:d + 1]), dt_bias=to_np(x.dt_bias[d:d + 1]), h0=sl(x.h0))


@pytest.mark.parametrize("name", ["scan_bf16_b8_d2048_l4096", "scan_bf16_b1_d5120_l65536_final_state"])
def test_bwd_full_size_sampled_channels(ssm, name):
    """The larger scan shapes at full size (the long one: 1024 time chunks):
    every output of 6 sampled channels (all batch rows), and the channel
    sums dA, dD, ddt_bias of those channels, against the oracle run on the
    channel alone."""
    w = I.WORKLOADS[name]
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], 1, io="bf16", recipe=w["recipe"],
                           seed=2, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(3)
    dy = torch.randn((w["batch"], w["dim"], w["seqlen"]), generator=g).to(torch.bfloat16).cuda()
    got = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    chans = sorted({0, w["dim"] - 1, *[int(v) for v in rng.integers(0, w["dim"], 4)]})
    for d in chans:
        ref = channel_slice_bwd(x, dy, d)
        for k in ("du", "ddelta", "dz"):
            e = rel_l2(to_np(got[k][:, d]), ref[k][:, 0])
            assert e <= TOL["bf16"][0], f"{name} d={d} {k}: rel_l2={e:.3e}"
        for k in ("dA", "dD", "ddt_bias", "dh0"):
            gk = to_np(got[k])[d] if k != "dh0" else to_np(got[k])[:, d]
            rk = ref[k][0] if k != "dh0" else ref[k][:, 0]
            e = rel_l2(gk, rk)
            assert e <= TOL["bf16"][1], f"{name} d={d} {k}: rel_l2={e:.3e}"


def test_autograd_function_matches_scan_bwd(ssm):
    """torch.autograd through selective_scan gives the library's gradients,
    including the final state's, in each input's dtype."""
    x = I.make_scan_inputs(2, 48, 16, 200, 2, io="bf16", recipe="scaled", seed=21, device="cuda", with_h0=True)
    leaves = {k: getattr(x, k).clone().requires_grad_(True) for k in ("u", "delta", "z", "A", "B", "C", "D",
                                                                        "dt_bias", "h0")}
    y, hf = ssm.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"], z=leaves["z"],
                               D=leaves["D"], dt_bias=leaves["dt_bias"], h0=leaves["h0"])
    g = torch.Generator(device="cpu").manual_seed(22)
    dy = torch.randn(y.shape, generator=g).to(y.dtype).cuda()
    dhf = torch.randn(hf.shape, generator=g).cuda()
    torch.autograd.backward([y, hf], [dy, dhf])
    ref = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0, dh_final=dhf)
    pairs = dict(u="du", delta="ddelta", z="dz", A="dA", B="dB", C="dC", D="dD", dt_bias="ddt_bias", h0="dh0")
    for k, r in pairs.items():
        got = leaves[k].grad
        assert got is not None and got.dtype == leaves[k].dtype, k
        assert rel_l2(to_np(got), to_np(ref[r].to(got.dtype))) <= 1e-6, k


def test_backward_writes_exactly_its_gradients(ssm):
    """Canary: every gradient is a view into a larger buffer filled with a
    sentinel (ragged L = 300 over three chunks, 70 channels, two groups, bf16);
    the kernels must write exactly the gradients' elements, and the values
    must match the oracle."""
    x = I.make_scan_inputs(1, 70 * 2, 16, 300, 2, io="bf16", recipe="scaled", seed=77, device="cuda", with_h0=True)
    dy = I.make_scan_inputs(1, 70 * 2, 16, 300, 2, io="bf16", recipe="scaled", seed=78, device="cuda").u
    batch, dim, L = x.u.shape
    N, G = x.A.shape[1], x.B.shape[1]
    shapes = dict(du=((batch, dim, L), torch.bfloat16), ddelta=((batch, dim, L), torch.bfloat16),
                  dz=((batch, dim, L), torch.bfloat16), dA=((dim, N), torch.float32),
                  dB=((batch, G, N, L), torch.float32), dC=((batch, G, N, L), torch.float32),
                  dD=((dim,), torch.float32), ddt_bias=((dim,), torch.float32), dh0=((batch, dim, N), torch.float32))
    pad = 2048
    bigs, out = {}, {}
    for k, (shape, dt) in shapes.items():
        n = int(np.prod(shape))
        bigs[k] = torch.full((n + 2 * pad,), 7.0, dtype=dt, device="cuda")
        out[k] = bigs[k][pad:pad + n].view(shape)
    gr = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0, out=out)
    torch.cuda.synchronize()
    for k, (shape, dt) in shapes.items():
        n = int(np.prod(shape))
        assert torch.all(bigs[k][:pad] == 7.0) and torch.all(bigs[k][pad + n:] == 7.0), k
    f = x.as_f64()
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], to_np(dy), z=f["z"], Dskip=f["Dskip"],
                          dt_bias=f["dt_bias"], h0=f["h0"])
    for k in ("du", "ddelta", "dz"):
        assert rel_l2(to_np(gr[k]), ref[k]) <= 5e-3, k
    for k in ("dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
        assert rel_l2(to_np(gr[k]), ref[k]) <= 1e-3, k
