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


def oracle_compare_blocks(x, y, hf=None, *, h0=None, block=256):
    """Compares a whole scan output y [batch, dim, L] (and h_final [batch,
    dim, N] when given) with the oracle, computed over blocks of ``block``
    channels so that host memory stays bounded on the largest workloads.
    Every element is compared: the rel-L2 sums are accumulated over the
    blocks, and fp32 max-rel uses the rms of the whole reference.  Returns
    (rel_l2_y, rel_l2_h or None, max_rel_y or None)."""
    batch, dim, L = x.u.shape
    G = x.B.shape[1]
    f64 = lambda t: None if t is None else t.detach().to("cpu", torch.float32).double().numpy()
    A, D, bias = f64(x.A), f64(x.D), f64(x.dt_bias)
    h0n = f64(h0) if h0 is not None else (f64(x.h0) if x.h0 is not None else None)
    num = den = hnum = hden = 0.0
    diffs, refs = [], []
    for d0 in range(0, dim, block):
        d1 = min(dim, d0 + block)
        if G == 1:
            gs = slice(0, 1)
        else:
            dpg = dim // G
            assert d0 // dpg == (d1 - 1) // dpg, "a block must stay inside one group"
            gs = slice(d0 // dpg, d0 // dpg + 1)
        sub = dict(u=f64(x.u[:, d0:d1]), delta=f64(x.delta[:, d0:d1]),
                   z=None if x.z is None else f64(x.z[:, d0:d1]), A=A[d0:d1], B=f64(x.B[:, gs]),
                   C=f64(x.C[:, gs]), Dskip=D[d0:d1], dt_bias=bias[d0:d1],
                   h0=None if h0n is None else h0n[:, d0:d1])
        out = oracle.scan(**sub, return_final_state=hf is not None)
        ry, rh = (out if hf is not None else (out, None))
        gy = f64(y[:, d0:d1])
        num += float(np.sum((gy - ry) ** 2))
        den += float(np.sum(ry * ry))
        if x.u.dtype == torch.float32:
            diffs.append(np.abs(gy - ry).ravel())
            refs.append(np.abs(ry).ravel())
        if hf is not None:
            gh = f64(hf[:, d0:d1])
            hnum += float(np.sum((gh - rh) ** 2))
            hden += float(np.sum(rh * rh))
    e_y = float(np.sqrt(num / den)) if den > 0 else float(np.sqrt(num))
    e_h = (float(np.sqrt(hnum / hden)) if hden > 0 else float(np.sqrt(hnum))) if hf is not None else None
    e_m = None
    if diffs:
        dd, rr = np.concatenate(diffs), np.concatenate(refs)
        rms = float(np.sqrt(den / rr.size)) if rr.size else 0.0
        e_m = float(np.max(dd / np.maximum(rr, MAX_REL_GUARD * rms if rms > 0 else 1e-30))) if rr.size else 0.0
    return e_y, e_h, e_m
