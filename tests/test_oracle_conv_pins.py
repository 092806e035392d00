"""Pins for the oracle of the short causal convolution in front of the scan:
a hand-worked fixture, a library routine (np.convolve), the impulse
response, causality, splitting a sequence with its history, the decode step
against the whole-sequence form, and the width-1 case.  A plausible slip
(reversed taps, a window shifted by one step, history ignored or read in the
wrong order, bias or silu dropped, the decode state shifted the wrong way)
fails at least one of them (tests/test_oracle_mutants.py plants each)."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def silu_ref(v):
    return v / (1.0 + np.exp(-v))


def numpy_conv(x, w, bias, x_prev=None, silu=True):
    """Per channel: np.convolve of [history, x] with the reversed taps, the
    outputs aligned with x (a library routine as the windowed sum)."""
    batch, dim, L = x.shape
    W = w.shape[1]
    out = np.empty_like(x)
    for b in range(batch):
        for d in range(dim):
            hist = np.zeros(W - 1) if x_prev is None else x_prev[b, d]
            seq = np.concatenate([hist, x[b, d]])
            full = np.convolve(seq, w[d][::-1])             # full[n] = sum_k w[k] seq[n-(W-1)+k]
            v = full[W - 1:W - 1 + L] + (0.0 if bias is None else bias[d])
            out[b, d] = silu_ref(v) if silu else v
    return out


def test_conv_hand_worked_golden():
    with open(os.path.join(GOLDEN, "hand_worked_conv.json")) as f:
        spec = json.load(f)
    env = {"exp": math.exp}
    for c in spec["cases"]:
        W, L = len(c["w"]), len(c["x"])
        x = np.array(c["x"], dtype=float).reshape(1, 1, L)
        prev = None if c["x_prev"] is None else np.array(c["x_prev"], dtype=float).reshape(1, 1, W - 1)
        out, last = oracle.causal_conv1d(x, np.array([c["w"]], dtype=float), np.array([c["bias"]], dtype=float),
                                         prev, silu=c["silu"], return_last=True)
        want = np.array([eval(e, {}, env) for e in c["expected"]])
        want_last = np.array([eval(e, {}, env) for e in c["expected_last"]])
        np.testing.assert_allclose(out.ravel(), want, rtol=1e-14, atol=1e-15, err_msg=c["name"])
        np.testing.assert_allclose(last.ravel(), want_last, rtol=0, atol=0, err_msg=c["name"])
    for c in spec["decode"]:
        W = len(c["w"])
        st, out = oracle.causal_conv1d_update(np.array(c["state"], dtype=float).reshape(1, 1, W - 1),
                                              np.array([[c["x"]]], dtype=float), np.array([c["w"]], dtype=float),
                                              np.array([c["bias"]], dtype=float), silu=c["silu"])
        assert out[0, 0] == pytest.approx(eval(c["expected"], {}, env), rel=1e-14)
        np.testing.assert_array_equal(st.ravel(), [eval(e, {}, env) for e in c["expected_state"]])


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("history", [False, True])
def test_conv_matches_numpy_convolve(W, silu, history):
    rng = np.random.default_rng(100 + 10 * W + 2 * silu + history)
    x = rng.standard_normal((2, 3, 37))
    w = rng.standard_normal((3, W))
    bias = rng.standard_normal(3)
    prev = rng.standard_normal((2, 3, W - 1)) if history else None
    got = oracle.causal_conv1d(x, w, bias, prev, silu=silu)
    np.testing.assert_allclose(got, numpy_conv(x, w, bias, prev, silu), rtol=1e-13, atol=1e-13)


def test_conv_impulse_response():
    """A unit impulse at time p reads the taps back in reverse order:
    out[p + j] = w[W-1-j] for j < W, zero elsewhere (no bias, no silu)."""
    W, L, p = 4, 12, 5
    w = np.array([[0.25, -1.5, 2.0, 3.0]])
    x = np.zeros((1, 1, L))
    x[0, 0, p] = 1.0
    out = oracle.causal_conv1d(x, w, None, silu=False).ravel()
    want = np.zeros(L)
    for j in range(W):
        want[p + j] = w[0, W - 1 - j]
    np.testing.assert_array_equal(out, want)


def test_conv_is_causal():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1, 2, 20))
    w = rng.standard_normal((2, 4))
    bias = rng.standard_normal(2)
    base = oracle.causal_conv1d(x, w, bias)
    x2 = x.copy()
    x2[:, :, 11] += 5.0
    moved = oracle.causal_conv1d(x2, w, bias)
    np.testing.assert_array_equal(moved[:, :, :11], base[:, :, :11])
    assert np.all(np.abs(moved[:, :, 11:15] - base[:, :, 11:15]) > 0)
    np.testing.assert_array_equal(moved[:, :, 15:], base[:, :, 15:])


@pytest.mark.parametrize("split", [1, 2, 3, 9, 19])
def test_conv_history_splits_sequence(split):
    """Convolving x[:s] and then x[s:] with the first part's last W-1 inputs
    as history equals convolving x in one piece."""
    rng = np.random.default_rng(11 + split)
    x = rng.standard_normal((2, 3, 20))
    w = rng.standard_normal((3, 4))
    bias = rng.standard_normal(3)
    prev = rng.standard_normal((2, 3, 3))
    whole, last = oracle.causal_conv1d(x, w, bias, prev, return_last=True)
    a, mid = oracle.causal_conv1d(x[:, :, :split], w, bias, prev, return_last=True)
    b, end = oracle.causal_conv1d(x[:, :, split:], w, bias, mid, return_last=True)
    np.testing.assert_allclose(np.concatenate([a, b], axis=2), whole, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(end, last)
    np.testing.assert_array_equal(last, x[:, :, -3:])


def test_conv_decode_steps_equal_conv():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 4, 16))
    w = rng.standard_normal((4, 3))
    bias = rng.standard_normal(4)
    prev = rng.standard_normal((3, 4, 2))
    whole, last = oracle.causal_conv1d(x, w, bias, prev, return_last=True)
    st = prev.copy()
    steps = []
    for t in range(16):
        st, o = oracle.causal_conv1d_update(st, x[:, :, t], w, bias)
        steps.append(o)
    np.testing.assert_allclose(np.stack(steps, axis=2), whole, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(st, last)


def test_conv_width_one_is_pointwise():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 5, 9))
    w = rng.standard_normal((5, 1))
    bias = rng.standard_normal(5)
    np.testing.assert_allclose(oracle.causal_conv1d(x, w, bias),
                               silu_ref(w[None, :, :] * x + bias[None, :, None]), rtol=1e-15, atol=1e-15)


def test_conv_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.causal_conv1d(np.zeros((1, 2, 4)), np.zeros((3, 4)))
    with pytest.raises(ValueError):
        oracle.causal_conv1d(np.zeros((1, 2, 4)), np.zeros((2, 4)), x_prev=np.zeros((1, 2, 4)))
