"""Pins of the fp64 oracle's backward pass (CPU only).

The backward pass is pinned against things other than itself:
- central finite differences of the forward oracle (itself pinned by
  test_oracle_pins.py) for every element of every input, on small cases with
  and without the gate, with several groups, an initial state and a gradient
  on the final state;
- the closed form of every gradient at L = 1, derived by hand from
  y = (sum_n C_n (Abar_n h0_n + Delta B_n u) + D u) * silu(z);
- the empty sequence, where h_final = h0 so that dh0 = dh_final.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

INPUTS = ("u", "delta", "z", "A", "B", "C", "Dskip", "dt_bias", "h0")
GRAD_OF = dict(u="du", delta="ddelta", z="dz", A="dA", B="dB", C="dC", Dskip="dD", dt_bias="ddt_bias", h0="dh0")


def case(rng, batch, dim, N, L, G, gated=True):
    c = dict(u=rng.standard_normal((batch, dim, L)), delta=rng.standard_normal((batch, dim, L)),
             z=rng.standard_normal((batch, dim, L)) if gated else None,
             A=-np.exp(0.5 * rng.standard_normal((dim, N))),
             B=rng.standard_normal((batch, G, N, L)), C=rng.standard_normal((batch, G, N, L)),
             Dskip=rng.standard_normal(dim), dt_bias=rng.standard_normal(dim),
             h0=rng.standard_normal((batch, dim, N)))
    return c


def loss(c, dy, dhf):
    y, hf = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                        dt_bias=c["dt_bias"], h0=c["h0"], return_final_state=True, nthreads=1)
    out = float(np.sum(y * dy))
    if dhf is not None:
        out += float(np.sum(hf * dhf))
    return out


def finite_difference(c, dy, dhf, name, eps=1e-6):
    x = c[name]
    g = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        keep = x[idx]
        x[idx] = keep + eps
        lp = loss(c, dy, dhf)
        x[idx] = keep - eps
        lm = loss(c, dy, dhf)
        x[idx] = keep
        g[idx] = (lp - lm) / (2 * eps)
    return g


@pytest.mark.parametrize("gated,with_dhf,G", [(True, True, 2), (False, False, 1), (True, False, 1)])
def test_gradients_match_finite_differences(gated, with_dhf, G):
    rng = np.random.default_rng(31 + 2 * G + gated)
    c = case(rng, 2, 4, 3, 6, G, gated)
    dy = rng.standard_normal(c["u"].shape)
    dhf = rng.standard_normal(c["h0"].shape) if with_dhf else None
    gr = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, z=c["z"], Dskip=c["Dskip"],
                         dt_bias=c["dt_bias"], h0=c["h0"], dh_final=dhf, nthreads=2)
    for name in INPUTS:
        if c[name] is None:
            assert gr[GRAD_OF[name]] is None
            continue
        fd = finite_difference(c, dy, dhf, name)
        an = gr[GRAD_OF[name]]
        scale = max(1.0, float(np.max(np.abs(fd))))
        err = float(np.max(np.abs(an - fd))) / scale
        assert err < 1e-7, f"d{name}: max error {err:.3e} against finite differences"


@pytest.mark.parametrize("gated", [False, True])
def test_single_step_closed_form(gated):
    rng = np.random.default_rng(5 + gated)
    c = case(rng, 1, 3, 4, 1, 1, gated)
    dy = rng.standard_normal(c["u"].shape)
    gr = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, z=c["z"], Dskip=c["Dskip"],
                         dt_bias=c["dt_bias"], h0=c["h0"], nthreads=1)
    for d in range(3):
        u, x = c["u"][0, d, 0], c["delta"][0, d, 0] + c["dt_bias"][d]
        dt = np.log1p(np.exp(x))
        sig = 1.0 / (1.0 + np.exp(-x))
        A, B, C, h0 = c["A"][d], c["B"][0, 0, :, 0], c["C"][0, 0, :, 0], c["h0"][0, d]
        a = np.exp(dt * A)
        h = a * h0 + dt * B * u
        s = C @ h + c["Dskip"][d] * u
        if gated:
            zv = c["z"][0, d, 0]
            sz = 1.0 / (1.0 + np.exp(-zv))
            g = dy[0, d, 0] * zv * sz
            dz = dy[0, d, 0] * s * sz * (1.0 + zv * (1.0 - sz))
            assert abs(gr["dz"][0, d, 0] - dz) < 1e-12 * max(1, abs(dz))
        else:
            g = dy[0, d, 0]
        dDelta = g * np.sum(C * (A * a * h0 + B * u))
        expect = dict(du=g * (dt * (C @ B) + c["Dskip"][d]), ddelta=dDelta * sig, dD=g * u, ddt_bias=dDelta * sig)
        got = dict(du=gr["du"][0, d, 0], ddelta=gr["ddelta"][0, d, 0], dD=gr["dD"][d], ddt_bias=gr["ddt_bias"][d])
        for k in expect:
            assert abs(got[k] - expect[k]) < 1e-12 * max(1, abs(expect[k])), k
        np.testing.assert_allclose(gr["dh0"][0, d], g * C * a, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(gr["dA"][d], g * C * h0 * a * dt, rtol=1e-12, atol=1e-14)
    # B and C are shared by the three channels of the group: their gradients sum over them.
    dB = np.zeros(4)
    dC = np.zeros(4)
    for d in range(3):
        u, x = c["u"][0, d, 0], c["delta"][0, d, 0] + c["dt_bias"][d]
        dt = np.log1p(np.exp(x))
        a = np.exp(dt * c["A"][d])
        g = dy[0, d, 0] * (c["z"][0, d, 0] / (1 + np.exp(-c["z"][0, d, 0])) if gated else 1.0)
        dB += g * c["C"][0, 0, :, 0] * dt * u
        dC += g * (a * c["h0"][0, d] + dt * c["B"][0, 0, :, 0] * u)
    np.testing.assert_allclose(gr["dB"][0, 0, :, 0], dB, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gr["dC"][0, 0, :, 0], dC, rtol=1e-12, atol=1e-14)


def test_empty_sequence_passes_dh_final_to_h0():
    rng = np.random.default_rng(9)
    c = case(rng, 2, 3, 4, 0, 1)
    dhf = rng.standard_normal(c["h0"].shape)
    gr = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], np.zeros(c["u"].shape), z=c["z"],
                         Dskip=c["Dskip"], dt_bias=c["dt_bias"], h0=c["h0"], dh_final=dhf)
    np.testing.assert_array_equal(gr["dh0"], dhf)
    assert not np.any(gr["dA"]) and not np.any(gr["dD"]) and not np.any(gr["ddt_bias"])


def test_threads_do_not_change_sums():
    rng = np.random.default_rng(4)
    c = case(rng, 3, 8, 4, 9, 2)
    dy = rng.standard_normal(c["u"].shape)
    kw = dict(z=c["z"], Dskip=c["Dskip"], dt_bias=c["dt_bias"], h0=c["h0"])
    g1 = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, nthreads=1, **kw)
    g5 = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, nthreads=5, **kw)
    for k, v in g1.items():
        np.testing.assert_allclose(g5[k], v, rtol=1e-13, atol=1e-13, err_msg=k)
