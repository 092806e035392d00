"""A correctly rounded fp32 evaluation of the selective scan, for tests.

This is not the oracle (the oracle is fp64, in ``oracle/``) and not the CUDA
path: it is the recurrence of eightmm.github.io "Mamba" (Main Claim, Scan View)
with the step size, decay and input term of intvml.com "DL0170 Mamba
Selective SSM vs Attention" (Mathematical Formulation), evaluated the way an
ideal fp32 kernel would: every product, sum and fused multiply-add rounded
once to fp32 (round to nearest even), every exponential and logarithm the
correctly rounded fp32 value of the exact function.  No fp32 evaluation of
the same sequence of operations can be more accurate, so its error against
the fp64 oracle is the floor that any fp32 kernel meets at best; the tests
use it to pin what the error metrics can demand of fp32 I/O.

It vectorises over (batch, channel, state) and walks time in a Python loop,
so it is meant for sequences of a few thousand steps at most.
"""
from __future__ import annotations

import numpy as np

f32 = np.float32


def _r(x):
    """Round fp64 values to fp32 (nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    """fp32 fused multiply-add: the fp64 product of two fp32 values is exact,
    so only the final sum rounds (twice: to fp64, then to fp32; the double
    rounding changes a result only in rare ties)."""
    return _r(np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64))


def exp32(x):
    return _r(np.exp(np.asarray(x, np.float64)))


def softplus32(v):
    """max(v, 0) + log1p(exp(-|v|)), each function correctly rounded to fp32."""
    v = np.asarray(v, np.float32)
    w = exp32(-np.abs(v))
    return _r(np.maximum(v, f32(0)).astype(np.float64) + _r(np.log1p(w.astype(np.float64))).astype(np.float64))


def silu32(z):
    z = np.asarray(z, np.float32)
    den = _r(f32(1).astype(np.float64) + exp32(-z).astype(np.float64))
    return _r(z.astype(np.float64) / den.astype(np.float64))


def scan_fp32(u, delta, A, B, C, z=None, Dskip=None, dt_bias=None, h0=None, return_final_state=False):
    """y [b, d, L] (fp32) of the selective scan, ungrouped or grouped (g = d / (dim / G)).

    Per step: Delta = softplus(delta + dt_bias); Abar = exp(Delta A);
    h = fma(Abar, h, (Delta u) B); y = fma(D, u, sum_n C h) * silu(z), the
    readout summed over n in order with fused multiply-adds."""
    u = np.asarray(u, np.float32)
    delta = np.asarray(delta, np.float32)
    A = np.asarray(A, np.float32)
    B = np.asarray(B, np.float32)
    C = np.asarray(C, np.float32)
    b_, d_, L = u.shape
    G, N = B.shape[1], B.shape[2]
    g_of_d = np.arange(d_) // (d_ // G)
    bias = np.zeros(d_, np.float32) if dt_bias is None else np.asarray(dt_bias, np.float32)
    dsk = np.zeros(d_, np.float32) if Dskip is None else np.asarray(Dskip, np.float32)
    h = np.zeros((b_, d_, N), np.float32) if h0 is None else np.asarray(h0, np.float32).copy()
    y = np.empty((b_, d_, L), np.float32)
    for t in range(L):
        v = _r(delta[:, :, t].astype(np.float64) + bias[None, :].astype(np.float64))
        dt = softplus32(v)                                               # [b, d]
        x = _r(dt[:, :, None].astype(np.float64) * A[None].astype(np.float64))
        abar = exp32(x)                                                  # [b, d, N]
        du = _r(dt.astype(np.float64) * u[:, :, t].astype(np.float64))   # [b, d]
        Bt = B[:, :, :, t][:, g_of_d]                                    # [b, d, N]
        Ct = C[:, :, :, t][:, g_of_d]
        bx = _r(du[:, :, None].astype(np.float64) * Bt.astype(np.float64))
        h = fma32(abar, h, bx)
        acc = np.zeros((b_, d_), np.float32)
        for n in range(N):
            acc = fma32(Ct[:, :, n], h[:, :, n], acc)
        yt = fma32(dsk[None, :], u[:, :, t], acc)
        if z is not None:
            yt = _r(yt.astype(np.float64) * silu32(np.asarray(z, np.float32)[:, :, t]).astype(np.float64))
        y[:, :, t] = yt
    if return_final_state:
        return y, h
    return y
