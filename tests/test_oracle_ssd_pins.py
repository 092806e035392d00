"""Pins of the fp64 SSD (Mamba-2) oracle, on the CPU.

The SSD layer is the selective recurrence with a scalar decay per head
(eightmm.github.io "Mamba", Relation to Mamba-2).  oracle.ssd computes it with
its own per-head loop; these tests pin it to things other than itself:

* the separately pinned selective-scan oracle, given the same problem with the
  per-head parameters spread over the head's channels (A[d, n] = A[h] for
  every n, delta and dt_bias of channel d = those of its head, Dskip likewise);
* the quadratic "duality" form, written out directly from the causal matrix
  mixer y_t = sum_{s<=t} C_t (prod_{j=s+1..t} Abar_j) Bbar_s x_s of the same
  section -- with a scalar decay, the mixer is (C_t . B_s) exp(A sum Delta)
  Delta_s, a masked attention-like matrix -- plus the initial state's term and
  the skip, then the gate;
* the final state's closed form, and L = 0.
"""
import numpy as np
import pytest

import oracle

rng_seed = 1234


def make(batch, nheads, headdim, N, L, G, seed, with_z=True, with_h0=True):
    rng = np.random.default_rng(seed)
    dim = nheads * headdim
    x = rng.standard_normal((batch, dim, L))
    delta = rng.standard_normal((batch, nheads, L))
    z = rng.standard_normal((batch, dim, L)) if with_z else None
    A = -np.exp(rng.uniform(np.log(0.5), np.log(8.0), nheads))
    B = rng.standard_normal((batch, G, N, L)) / np.sqrt(N)
    C = rng.standard_normal((batch, G, N, L)) / np.sqrt(N)
    D = 1.0 + 0.1 * rng.standard_normal(nheads)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), nheads))
    dt_bias = np.log(np.expm1(dt))
    h0 = rng.standard_normal((batch, dim, N)) if with_h0 else None
    return dict(x=x, delta=delta, z=z, A=A, B=B, C=C, Dskip=D, dt_bias=dt_bias, h0=h0)


def spread(p, headdim):
    """The same problem for the per-channel scan: head parameters repeated over
    the head's channels."""
    N = p["B"].shape[2]
    rep = lambda v: np.repeat(v, headdim, axis=-1)
    return dict(u=p["x"], delta=np.repeat(p["delta"], headdim, axis=1), z=p["z"],
                A=np.repeat(p["A"], headdim)[:, None] * np.ones((1, N)), B=p["B"], C=p["C"],
                Dskip=rep(p["Dskip"]), dt_bias=rep(p["dt_bias"]), h0=p["h0"])


def softplus(v):
    return np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))


def quadratic(p, headdim):
    """y from the causal matrix-mixer (duality) form, O(L^2) per head."""
    x, delta, z, A, B, C = p["x"], p["delta"], p["z"], p["A"], p["B"], p["C"]
    batch, dim, L = x.shape
    nheads = dim // headdim
    G = B.shape[1]
    y = np.zeros_like(x)
    for b in range(batch):
        for h in range(nheads):
            g = h // (nheads // G)
            dt = softplus(delta[b, h] + p["dt_bias"][h])           # [L]
            S = np.concatenate([[0.0], np.cumsum(dt)])              # S[t+1] = sum_{j<=t} Delta_j
            CB = C[b, g].T @ B[b, g]                                # [L, L]: C_t . B_s
            dec = np.exp(A[h] * (S[1:, None] - S[None, 1:]))        # exp(A sum_{j=s+1..t} Delta_j)
            Mx = np.tril(CB * dec) * dt[None, :]                    # mixer with Bbar = Delta B
            xs = x[b, h * headdim:(h + 1) * headdim]                # [P, L]
            yh = xs @ Mx.T                                          # y_t[p] = sum_s M[t,s] x_s[p]
            if p["h0"] is not None:
                h0 = p["h0"][b, h * headdim:(h + 1) * headdim]      # [P, N]
                yh += (h0 @ C[b, g]) * np.exp(A[h] * S[1:])[None, :]
            yh += p["Dskip"][h] * xs
            if z is not None:
                zz = z[b, h * headdim:(h + 1) * headdim]
                yh *= zz / (1 + np.exp(-zz))
            y[b, h * headdim:(h + 1) * headdim] = yh
    return y


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("with_z", [True, False])
def test_ssd_equals_the_scan_with_spread_parameters(G, with_z):
    p = make(2, 4, 3, 8, 37, G, seed=1, with_z=with_z)
    y, hf = oracle.ssd(**p, headdim=3, return_final_state=True)
    ry, rh = oracle.scan(**spread(p, 3), return_final_state=True)
    assert np.max(np.abs(y - ry)) < 1e-12 * max(1.0, np.max(np.abs(ry)))
    assert np.max(np.abs(hf - rh)) < 1e-12 * max(1.0, np.max(np.abs(rh)))


@pytest.mark.parametrize("G", [1, 2])
def test_ssd_equals_the_quadratic_duality_form(G):
    p = make(1, 4, 5, 6, 48, G, seed=2)
    y = oracle.ssd(**p, headdim=5)
    q = quadratic(p, 5)
    assert np.max(np.abs(y - q)) < 1e-11 * max(1.0, np.max(np.abs(q)))


def test_ssd_final_state_closed_form():
    p = make(1, 2, 4, 5, 30, 1, seed=3, with_z=False)
    _, hf = oracle.ssd(**p, headdim=4, return_final_state=True)
    for h in range(2):
        dt = softplus(p["delta"][0, h] + p["dt_bias"][h])
        tail = np.concatenate([np.cumsum(dt[::-1])[::-1][1:], [0.0]])  # sum_{j>s} Delta_j
        w = np.exp(p["A"][h] * tail) * dt                               # [L]
        xs = p["x"][0, h * 4:(h + 1) * 4]                                # [P, L]
        want = np.exp(p["A"][h] * dt.sum()) * p["h0"][0, h * 4:(h + 1) * 4] + (xs * w) @ p["B"][0, 0].T
        assert np.max(np.abs(hf[0, h * 4:(h + 1) * 4] - want)) < 1e-12 * np.max(np.abs(want))


def test_ssd_empty_sequence_returns_h0():
    p = make(1, 2, 2, 4, 0, 1, seed=4)
    y, hf = oracle.ssd(**p, headdim=2, return_final_state=True)
    assert y.shape == (1, 4, 0)
    assert np.array_equal(hf, p["h0"])


def test_ssd_rejects_bad_groups():
    p = make(1, 3, 2, 4, 5, 1, seed=5)
    p["B"] = np.repeat(p["B"], 2, axis=1)
    p["C"] = np.repeat(p["C"], 2, axis=1)
    with pytest.raises(ValueError):
        oracle.ssd(**p, headdim=2)  # 3 heads do not split into 2 groups
