"""Helpers for the GPU-vs-oracle parity tests: error metrics, tolerances and
running the oracle on exactly the values the GPU saw."""
import numpy as np
import torch

import oracle

# Tolerances (fp32 I/O: rel-L2 and guarded max-rel; bf16 I/O with fp32 state:
# rel-L2 against the oracle run on the same bf16-rounded inputs).
F32_REL_L2 = 1e-5
F32_MAX_REL = 1e-4
BF16_REL_L2 = 5e-3
STATE_REL_L2 = 1e-4


def to_np(t):
    return t.detach().to("cpu", torch.float32).double().numpy()


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den > 0 else 1.0))


MAX_REL_GUARD = 1e-2


def max_rel(x, ref, guard=MAX_REL_GUARD):
    """max |x - r| / max(|r|, guard * rms(r)).  The guard keeps outputs that
    sit near zero -- silu(z ~ 0), or cancellation among the terms of C.h --
    from turning the fp32 rounding floor (~1e-7 of the terms) into a huge
    relative error; a correctly rounded fp32 evaluation of the recurrence
    already exceeds 1e-4 with a guard of 1e-3 rms."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), guard * rms if rms > 0 else 1e-30)
    return float(np.max(np.abs(x - ref) / den))


def assert_close(y, ref, io, what=""):
    e2 = rel_l2(y, ref)
    if io == "f32":
        em = max_rel(y, ref)
        assert e2 <= F32_REL_L2 and em <= F32_MAX_REL, f"{what}: rel_l2={e2:.3e} max_rel={em:.3e}"
    else:
        assert e2 <= BF16_REL_L2, f"{what}: rel_l2={e2:.3e}"
    return e2


def oracle_scan(x, *, h0=None, final_state=False, channels=None, nthreads=None):
    """Oracle on the inputs held by ScanInputs x (any device).  ``channels`` =
    optional list of (b, d) pairs: then only those rows are computed and the
    result is [len(channels), L] (requires ngroups == 1)."""
    f = x.as_f64()
    if h0 is not None:
        f["h0"] = to_np(h0)
    if channels is None:
        return oracle.scan(**f, return_final_state=final_state, nthreads=nthreads)
    assert f["B"].shape[1] == 1
    ys, hs = [], []
    for b, d in channels:
        sub = dict(u=f["u"][b:b + 1, d:d + 1], delta=f["delta"][b:b + 1, d:d + 1],
                   z=None if f["z"] is None else f["z"][b:b + 1, d:d + 1],
                   A=f["A"][d:d + 1], B=f["B"][b:b + 1], C=f["C"][b:b + 1],
                   Dskip=f["Dskip"][d:d + 1], dt_bias=f["dt_bias"][d:d + 1],
                   h0=None if f["h0"] is None else f["h0"][b:b + 1, d:d + 1])
        out = oracle.scan(**sub, return_final_state=final_state, nthreads=1)
        if final_state:
            ys.append(out[0][0, 0])
            hs.append(out[1][0, 0])
        else:
            ys.append(out[0, 0])
    if final_state:
        return np.stack(ys), np.stack(hs)
    return np.stack(ys)
