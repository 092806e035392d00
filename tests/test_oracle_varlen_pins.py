"""Pins for the oracle of packed variable-length batches and of the decode
step on a pool of state slots.  The packed scan must equal the (separately
pinned) scan run on each sequence alone from its own h0; sequences must not
see each other; an empty sequence returns its h0.  The pooled decode step must
equal the plain decode step on the gathered states, touch no other slot and
skip padding rows.  Planted slips (no reset between sequences, every sequence
starting from the first one's h0, the wrong group, the pooled step reading the
batch row's slot) are each caught (tests/test_oracle_mutants.py)."""
import numpy as np
import pytest

import oracle


def varlen_case(rng, dim=6, N=4, G=2, cu=(0, 7, 7, 19, 20, 33)):
    T = cu[-1]
    nseq = len(cu) - 1
    return dict(
        u=rng.standard_normal((dim, T)), delta=rng.standard_normal((dim, T)), z=rng.standard_normal((dim, T)),
        A=-np.exp(rng.uniform(-1.0, 1.0, (dim, N))), B=rng.standard_normal((G, N, T)),
        C=rng.standard_normal((G, N, T)), Dskip=rng.standard_normal(dim), dt_bias=rng.uniform(-3.0, -1.0, dim),
        h0=rng.standard_normal((nseq, dim, N)), cu_seqlens=np.array(cu, dtype=np.int32))


def per_sequence(c):
    """The scan oracle on each sequence alone (batch 1), from its own h0."""
    cu = c["cu_seqlens"]
    dim, T = c["u"].shape
    N = c["A"].shape[1]
    y = np.zeros((dim, T))
    hf = np.zeros((len(cu) - 1, dim, N))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if b == a:
            hf[s] = c["h0"][s]
            continue
        ys, hs = oracle.scan(c["u"][None, :, a:b], c["delta"][None, :, a:b], c["A"], c["B"][None, :, :, a:b],
                             c["C"][None, :, :, a:b], z=c["z"][None, :, a:b], Dskip=c["Dskip"],
                             dt_bias=c["dt_bias"], h0=c["h0"][s][None], return_final_state=True)
        y[:, a:b] = ys[0]
        hf[s] = hs[0]
    return y, hf


def test_varlen_equals_each_sequence_alone():
    c = varlen_case(np.random.default_rng(0))
    y, hf = oracle.scan_varlen(**c, return_final_state=True)
    ry, rh = per_sequence(c)
    np.testing.assert_allclose(y, ry, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hf, rh, rtol=1e-13, atol=1e-13)


def test_varlen_sequences_do_not_see_each_other():
    c = varlen_case(np.random.default_rng(1))
    y = oracle.scan_varlen(**c)
    c2 = dict(c)
    c2["u"] = c["u"].copy()
    c2["u"][:, 8:19] += 3.0   # tokens of sequence 2 only
    y2 = oracle.scan_varlen(**c2)
    np.testing.assert_array_equal(y2[:, :8], y[:, :8])
    np.testing.assert_array_equal(y2[:, 19:], y[:, 19:])
    assert np.all(np.abs(y2[:, 8:19] - y[:, 8:19]).max(axis=1) > 0)


def test_varlen_single_sequence_is_the_scan():
    c = varlen_case(np.random.default_rng(2), cu=(0, 25))
    y, hf = oracle.scan_varlen(**c, return_final_state=True)
    ry, rh = per_sequence(c)
    np.testing.assert_allclose(y, ry, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hf, rh, rtol=1e-13, atol=1e-13)


def test_varlen_empty_sequence_returns_its_h0():
    c = varlen_case(np.random.default_rng(3))
    _, hf = oracle.scan_varlen(**c, return_final_state=True)
    np.testing.assert_array_equal(hf[1], c["h0"][1])   # sequence 1 is [7, 7)


def test_varlen_padding_after_the_last_sequence_is_not_read():
    """A row longer than the packed sequences: the trailing times are padding."""
    c = varlen_case(np.random.default_rng(6))
    y, hf = oracle.scan_varlen(**c, return_final_state=True)
    T = c["u"].shape[1]
    pad = {k: (np.concatenate([v, 100.0 + np.zeros(v.shape[:-1] + (5,))], axis=-1)
               if k in ("u", "delta", "z", "B", "C") else v) for k, v in c.items()}
    y2, hf2 = oracle.scan_varlen(**pad, return_final_state=True)
    np.testing.assert_array_equal(y2[:, :T], y)
    np.testing.assert_array_equal(hf2, hf)


def test_varlen_rejects_bad_offsets():
    c = varlen_case(np.random.default_rng(4))
    for bad in ([0, 7, 5, 19, 20, 33], [1, 7, 7, 19, 20, 33], [0, 7, 7, 19, 20, 34]):
        with pytest.raises(ValueError):
            oracle.scan_varlen(**dict(c, cu_seqlens=np.array(bad, dtype=np.int32)))


def test_pooled_decode_equals_gathered_decode():
    rng = np.random.default_rng(5)
    slots, batch, dim, N, G = 7, 5, 6, 4, 2
    pool = rng.standard_normal((slots, dim, N))
    idx = np.array([3, -1, 0, 6, 2], dtype=np.int32)
    tok = dict(u=rng.standard_normal((batch, dim)), delta=rng.standard_normal((batch, dim)),
               z=rng.standard_normal((batch, dim)), B=rng.standard_normal((batch, G, N)),
               C=rng.standard_normal((batch, G, N)))
    A = -np.exp(rng.uniform(-1.0, 1.0, (dim, N)))
    Dskip, dt_bias = rng.standard_normal(dim), rng.uniform(-3.0, -1.0, dim)
    new, y = oracle.state_update_indexed(pool, idx, tok["u"], tok["delta"], A, tok["B"], tok["C"], z=tok["z"],
                                         Dskip=Dskip, dt_bias=dt_bias)
    live = idx >= 0
    st, ry = oracle.state_update(pool[idx[live]], tok["u"][live], tok["delta"][live], A, tok["B"][live],
                                 tok["C"][live], z=tok["z"][live], Dskip=Dskip, dt_bias=dt_bias)
    np.testing.assert_allclose(y[live], ry, rtol=1e-14, atol=1e-14)
    assert np.all(np.isnan(y[~live]))
    np.testing.assert_allclose(new[idx[live]], st, rtol=1e-14, atol=1e-14)
    untouched = np.setdiff1d(np.arange(slots), idx[live])
    np.testing.assert_array_equal(new[untouched], pool[untouched])
