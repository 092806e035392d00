"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a hand-worked example, a closed form, an O(L^2) brute-force sum, a
library routine (np.convolve, np.logaddexp) or a limit that the pages fix.

A plausible slip in the oracle (dropped skip term, wrong sign of A, B and C
swapped in time, wrong group index, bias added after softplus, gate applied to
the state instead of the output, lost initial state) fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def softplus_ref(x):
    return np.logaddexp(0.0, x)  # log(e^0 + e^x), a library routine


def silu_ref(z):
    return z / (1.0 + np.exp(-z))


def rand_case(rng, batch, dim, N, L, G, *, delta_scale=1.0):
    return dict(
        u=rng.standard_normal((batch, dim, L)),
        delta=delta_scale * rng.standard_normal((batch, dim, L)),
        z=rng.standard_normal((batch, dim, L)),
        A=-np.exp(rng.uniform(-1.0, 1.5, (dim, N))),
        B=rng.standard_normal((batch, G, N, L)),
        C=rng.standard_normal((batch, G, N, L)),
        Dskip=rng.standard_normal(dim),
        dt_bias=rng.uniform(-4.0, -1.0, dim),
        h0=rng.standard_normal((batch, dim, N)),
    )


def brute_force_mixer(c, with_h0=True, gated=True):
    """Causal matrix-mixer expansion of the selective recurrence
    (eightmm.github.io "Mamba", Relation to Mamba-2):
        y_t = sum_{i<=t} C_t (prod_{j=i+1..t} Abar_j) Bbar_i x_i,
    written with exponent sums, O(L^2) per channel, plus the h0 term
    C_t (prod_{j=1..t} Abar_j) h0 and the skip / gate of the readout."""
    u, delta, A, B, C = c["u"], c["delta"], c["A"], c["B"], c["C"]
    batch, dim, L = u.shape
    G = B.shape[1]
    y = np.zeros_like(u)
    for b in range(batch):
        for d in range(dim):
            g = d // (dim // G)
            dt = softplus_ref(delta[b, d] + c["dt_bias"][d])       # [L]
            S = np.cumsum(dt)                                       # S_t = sum_{j<=t} Delta_j
            for t in range(L):
                acc = 0.0
                for i in range(t + 1):
                    decay = np.exp(A[d] * (S[t] - S[i]))            # prod_{j=i+1..t} Abar_j, [N]
                    acc += np.sum(C[b, g, :, t] * decay * dt[i] * B[b, g, :, i]) * u[b, d, i]
                if with_h0:
                    acc += np.sum(C[b, g, :, t] * np.exp(A[d] * S[t]) * c["h0"][b, d])
                yt = acc + c["Dskip"][d] * u[b, d, t]
                if gated:
                    yt *= silu_ref(c["z"][b, d, t])
                y[b, d, t] = yt
    return y


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------
# Hand-worked golden cases
# --------------------------------------------------------------------------

def test_hand_worked_golden_cases():
    with open(os.path.join(GOLDEN, "hand_worked_n1.json")) as f:
        spec = json.load(f)
    env = {"ln2": math.log(2.0)}
    for case in spec["cases"]:
        L = len(case["u"])
        args = dict(
            u=np.array(case["u"]).reshape(1, 1, L),
            delta=np.array(case["delta"]).reshape(1, 1, L),
            A=np.array(case["A"]),
            B=np.array(case["B"]).reshape(1, 1, 1, L),
            C=np.array(case["C"]).reshape(1, 1, 1, L),
            z=None if case["z"] is None else np.array(case["z"]).reshape(1, 1, L),
            Dskip=np.array([case["D"]]),
            dt_bias=np.array([case["dt_bias"]]),
        )
        y, hf = oracle.scan(**args, return_final_state=True)
        want_y = np.array([eval(e, {}, env) for e in case["expected_y"]])
        want_h = np.array([eval(e, {}, env) for e in case["expected_h_final"]])
        np.testing.assert_allclose(y.ravel(), want_y, rtol=1e-14, atol=1e-15, err_msg=case["name"])
        np.testing.assert_allclose(hf.ravel(), want_h, rtol=1e-14, atol=1e-15, err_msg=case["name"])


def test_oracle_regression_fixture():
    """Frozen oracle output (written by tests/golden/make_oracle_regression.py)."""
    path = os.path.join(GOLDEN, "oracle_regression_small.json")
    with open(path) as f:
        spec = json.load(f)
    from selective_state_space_109_b300 import inputs as I
    x = I.make_scan_inputs(**spec["inputs"]).as_f64()
    y, hf = oracle.scan(**x, return_final_state=True)
    np.testing.assert_allclose(y.ravel()[: len(spec["y_head"])], spec["y_head"], rtol=1e-12)
    np.testing.assert_allclose(float(np.sum(y)), spec["y_sum"], rtol=1e-12)
    np.testing.assert_allclose(float(np.sum(hf * hf)), spec["h_final_sumsq"], rtol=1e-12)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gated", [False, True])
def test_single_step_closed_form(gated):
    """L = 1 from h0 = 0: y = C.(Delta B u) + D u, times silu(z) when gated."""
    rng = np.random.default_rng(1)
    c = rand_case(rng, 2, 6, 8, 1, 2)
    if not gated:
        c["z"] = None
    y = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                    dt_bias=c["dt_bias"])
    for b in range(2):
        for d in range(6):
            g = d // 3
            dt = softplus_ref(c["delta"][b, d, 0] + c["dt_bias"][d])
            want = np.dot(c["C"][b, g, :, 0], dt * c["B"][b, g, :, 0] * c["u"][b, d, 0]) \
                + c["Dskip"][d] * c["u"][b, d, 0]
            if gated:
                want *= silu_ref(c["z"][b, d, 0])
            assert abs(y[b, d, 0] - want) <= 1e-14 * max(1.0, abs(want))


def test_geometric_series_n1_constant_inputs():
    """N = 1, constant Delta, B = C = u = 1, h0 = 0:
    h_t = Delta (1 - a^t) / (1 - a) with a = exp(Delta A)."""
    L = 200
    for bias, Aval in [(-3.0, -1.0), (-6.0, -0.5), (0.5, -2.0)]:
        dt = float(softplus_ref(bias))
        a = math.exp(dt * Aval)
        y, hf = oracle.scan(np.ones((1, 1, L)), np.zeros((1, 1, L)), np.array([[Aval]]),
                            np.ones((1, 1, 1, L)), np.ones((1, 1, 1, L)), Dskip=np.array([0.7]),
                            dt_bias=np.array([bias]), return_final_state=True)
        t = np.arange(1, L + 1)
        want = dt * (1.0 - a ** t) / (1.0 - a) + 0.7
        np.testing.assert_allclose(y[0, 0], want, rtol=1e-12)
        np.testing.assert_allclose(hf[0, 0, 0], want[-1] - 0.7, rtol=1e-12)


# --------------------------------------------------------------------------
# Brute force (causal matrix mixer) with time-varying selective parameters
# --------------------------------------------------------------------------

@pytest.mark.parametrize("with_h0,gated", [(False, True), (True, True), (True, False)])
def test_matches_causal_matrix_mixer(with_h0, gated):
    rng = np.random.default_rng(2)
    c = rand_case(rng, 2, 4, 5, 37, 2)
    y = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"] if gated else None,
                    Dskip=c["Dskip"], dt_bias=c["dt_bias"], h0=c["h0"] if with_h0 else None)
    want = brute_force_mixer(c, with_h0=with_h0, gated=gated)
    assert rel_err(y, want) < 1e-12


def test_matches_causal_matrix_mixer_large_state():
    """N = 64 states (the large-state case of the library): the same
    brute-force causal matrix-mixer expansion."""
    rng = np.random.default_rng(12)
    c = rand_case(rng, 1, 3, 64, 13, 1)
    y = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                    dt_bias=c["dt_bias"], h0=c["h0"])
    assert rel_err(y, brute_force_mixer(c, with_h0=True, gated=True)) < 1e-12


def test_groups_read_their_own_B_C():
    """With G = 4 groups of 2 channels, each channel must use its group's B/C:
    the brute force indexes g = d // (dim / G) independently."""
    rng = np.random.default_rng(3)
    c = rand_case(rng, 1, 8, 4, 12, 4)
    y = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                    dt_bias=c["dt_bias"], h0=c["h0"])
    assert rel_err(y, brute_force_mixer(c)) < 1e-12
    # and swapping two groups' B changes exactly the channels of those groups
    c2 = dict(c)
    c2["B"] = c["B"][:, [1, 0, 2, 3]]
    y2 = oracle.scan(c2["u"], c2["delta"], c2["A"], c2["B"], c2["C"], z=c2["z"],
                     Dskip=c2["Dskip"], dt_bias=c2["dt_bias"], h0=c2["h0"])
    changed = np.any(np.abs(y2 - y) > 1e-12, axis=2)[0]
    assert changed.tolist() == [True] * 4 + [False] * 4


# --------------------------------------------------------------------------
# LTI special case == convolution (cuishuaiwen.com "Mamba & State-Space
# Sequence Models", Core mechanics / Self-check; intvml.com, point (3))
# --------------------------------------------------------------------------

def test_time_invariant_case_is_a_convolution():
    rng = np.random.default_rng(4)
    N, L = 6, 90
    A = -np.exp(rng.uniform(-1.0, 1.0, (1, N)))
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    u = rng.standard_normal(L)
    bias, D = -2.3, 0.4
    y = oracle.scan(u.reshape(1, 1, L), np.zeros((1, 1, L)), A,
                    np.tile(Bn[:, None], (1, 1, 1, L)).reshape(1, 1, N, L),
                    np.tile(Cn[:, None], (1, 1, 1, L)).reshape(1, 1, N, L),
                    Dskip=np.array([D]), dt_bias=np.array([bias]))
    dt = float(softplus_ref(bias))
    k = np.arange(L)
    kernel = np.sum(Cn[:, None] * np.power(np.exp(dt * A[0])[:, None], k[None, :]) * dt * Bn[:, None], axis=0)
    want = np.convolve(u, kernel)[:L] + D * u
    np.testing.assert_allclose(y[0, 0], want, rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------
# Limits of the step size (intvml.com, point (2): Delta acts as a forget gate)
# --------------------------------------------------------------------------

def test_vanishing_step_leaves_only_skip_path():
    """dt_bias = -60: Delta ~ 1e-26, the state stays ~0, y = D u silu(z)."""
    rng = np.random.default_rng(5)
    c = rand_case(rng, 1, 3, 16, 64, 1)
    y = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                    dt_bias=np.full(3, -60.0))
    want = c["Dskip"][None, :, None] * c["u"] * silu_ref(c["z"])
    assert rel_err(y, want) < 1e-14


def test_tiny_step_ignores_one_token():
    """A single step with Delta ~ 0 leaves the state as it was (the token is skipped)."""
    rng = np.random.default_rng(6)
    c = rand_case(rng, 1, 2, 8, 20, 1)
    c["delta"][0, :, 10] = -80.0
    _, h10 = oracle.scan(c["u"][..., :10], c["delta"][..., :10], c["A"], c["B"][..., :10],
                         c["C"][..., :10], dt_bias=c["dt_bias"], return_final_state=True)
    _, h11 = oracle.scan(c["u"][..., :11], c["delta"][..., :11], c["A"], c["B"][..., :11],
                         c["C"][..., :11], dt_bias=c["dt_bias"], return_final_state=True)
    np.testing.assert_allclose(h11, h10, rtol=1e-15, atol=1e-30)


def test_large_step_overwrites_state():
    """delta + dt_bias = 50 and A <= -1: Abar < e^-50, so h_t = Delta B_t u_t and
    y_t = Delta (C_t . B_t) u_t + D u_t, whatever came before."""
    rng = np.random.default_rng(7)
    c = rand_case(rng, 1, 3, 8, 40, 1)
    A = -1.0 - np.abs(c["A"])
    y = oracle.scan(c["u"], np.zeros_like(c["u"]), A, c["B"], c["C"], Dskip=c["Dskip"],
                    dt_bias=np.full(3, 50.0), h0=c["h0"])
    dt = float(softplus_ref(50.0))
    cb = np.sum(c["C"][0, 0] * c["B"][0, 0], axis=0)  # [L]
    want = dt * cb[None, :] * c["u"][0] + c["Dskip"][:, None] * c["u"][0]
    np.testing.assert_allclose(y[0], want, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Structure: linearity, split carry, decode == scan
# --------------------------------------------------------------------------

def test_ungated_output_is_linear_in_u_and_h0():
    rng = np.random.default_rng(8)
    c1 = rand_case(rng, 1, 3, 8, 30, 1)
    c2 = rand_case(rng, 1, 3, 8, 30, 1)
    common = dict(A=c1["A"], B=c1["B"], C=c1["C"], Dskip=c1["Dskip"], dt_bias=c1["dt_bias"])
    f = lambda u, h0: oracle.scan(u, c1["delta"], common["A"], common["B"], common["C"],
                                  Dskip=common["Dskip"], dt_bias=common["dt_bias"], h0=h0)
    y1, y2 = f(c1["u"], c1["h0"]), f(c2["u"], c2["h0"])
    y12 = f(2.0 * c1["u"] - 3.0 * c2["u"], 2.0 * c1["h0"] - 3.0 * c2["h0"])
    assert rel_err(y12, 2.0 * y1 - 3.0 * y2) < 1e-12


@pytest.mark.parametrize("split", [1, 17, 63])
def test_split_sequence_with_carried_state(split):
    rng = np.random.default_rng(9)
    c = rand_case(rng, 2, 3, 8, 64, 1)
    kw = dict(Dskip=c["Dskip"], dt_bias=c["dt_bias"])
    y, hf = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], h0=c["h0"],
                        return_final_state=True, **kw)
    s = split
    ya, ha = oracle.scan(c["u"][..., :s], c["delta"][..., :s], c["A"], c["B"][..., :s],
                         c["C"][..., :s], z=c["z"][..., :s], h0=c["h0"], return_final_state=True, **kw)
    yb, hb = oracle.scan(c["u"][..., s:], c["delta"][..., s:], c["A"], c["B"][..., s:],
                         c["C"][..., s:], z=c["z"][..., s:], h0=ha, return_final_state=True, **kw)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=2), y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hb, hf, rtol=1e-12, atol=1e-14)


def test_decode_steps_equal_one_scan():
    """Running state_update token by token equals one scan with the same h0
    (cuishuaiwen.com: inference uses the recurrence, O(1) per step)."""
    rng = np.random.default_rng(10)
    c = rand_case(rng, 2, 4, 8, 25, 2)
    y, hf = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], z=c["z"], Dskip=c["Dskip"],
                        dt_bias=c["dt_bias"], h0=c["h0"], return_final_state=True)
    st = c["h0"].copy()
    for t in range(25):
        st, yt = oracle.state_update(st, c["u"][..., t], c["delta"][..., t], c["A"],
                                     c["B"][..., t], c["C"][..., t], z=c["z"][..., t],
                                     Dskip=c["Dskip"], dt_bias=c["dt_bias"])
        np.testing.assert_allclose(yt, y[..., t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st, hf, rtol=1e-12, atol=1e-14)


def test_decode_single_step_from_zero_state():
    """One decode step from a zero state is the L = 1 closed form."""
    rng = np.random.default_rng(11)
    c = rand_case(rng, 3, 4, 8, 1, 1)
    st, y = oracle.state_update(np.zeros((3, 4, 8)), c["u"][..., 0], c["delta"][..., 0], c["A"],
                                c["B"][..., 0], c["C"][..., 0], z=c["z"][..., 0],
                                Dskip=c["Dskip"], dt_bias=c["dt_bias"])
    for b in range(3):
        for d in range(4):
            dt = softplus_ref(c["delta"][b, d, 0] + c["dt_bias"][d])
            np.testing.assert_allclose(st[b, d], dt * c["B"][b, 0, :, 0] * c["u"][b, d, 0], rtol=1e-14)
            want = (np.dot(c["C"][b, 0, :, 0], st[b, d]) + c["Dskip"][d] * c["u"][b, d, 0]) \
                * silu_ref(c["z"][b, d, 0])
            assert abs(y[b, d] - want) <= 1e-14 * max(1.0, abs(want))


def test_threads_do_not_change_results():
    rng = np.random.default_rng(12)
    c = rand_case(rng, 3, 5, 4, 33, 1)
    args = (c["u"], c["delta"], c["A"], c["B"], c["C"])
    kw = dict(z=c["z"], Dskip=c["Dskip"], dt_bias=c["dt_bias"], h0=c["h0"])
    y1 = oracle.scan(*args, nthreads=1, **kw)
    y4 = oracle.scan(*args, nthreads=4, **kw)
    assert np.array_equal(y1, y4)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.scan(np.zeros((1, 3, 4)), np.zeros((1, 3, 4)), np.zeros((3, 2)),
                    np.zeros((1, 2, 2, 4)), np.zeros((1, 2, 2, 4)))  # 3 channels, 2 groups
