"""fp64 CPU oracle for the selective scan (S6) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it, and it loads nothing of theirs.

The arithmetic lives in ``ssm_oracle.c`` (plain C, double precision, one
sequential recurrence per channel).  This module only compiles it with gcc on
first use and marshals numpy arrays to it.  See ``ssm_oracle.c`` for the
formulas and the passages of the pages they follow.

Pin status: every function here is pinned -- the scan and its decode step by
``tests/test_oracle_pins.py`` against closed forms, brute-force sums and limits
that the pages fix, the short causal convolution and its decode step by
``tests/test_oracle_conv_pins.py`` against a hand-worked fixture, np.convolve,
the impulse response and its split and decode identities, the packed
variable-length scan and the pooled decode step by
``tests/test_oracle_varlen_pins.py`` against the separately pinned scan and
decode step, the backward pass by ``tests/test_oracle_bwd_pins.py`` against
central finite differences of the pinned forward scan and a closed form at
L = 1, the SSD (Mamba-2) layer by ``tests/test_oracle_ssd_pins.py`` against
the separately pinned scan with its per-head parameters spread over the
channels and against the quadratic (matrix-mixer) form -- and
``tests/test_oracle_mutants.py`` checks that the pins catch planted slips.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into libssm_oracle.so next to it (gcc, -O2)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        # -ffp-contract=off: no fused multiply-adds, so each product and sum
        # rounds exactly as written in the C source.
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_scan.argtypes = [P] * 11 + [I] * 6
            lib.oracle_scan.restype = I
            lib.oracle_state_update.argtypes = [P] * 10 + [I] * 4
            lib.oracle_state_update.restype = I
            _set_conv_types(lib)
            _lib = lib
    return _lib


def _set_conv_types(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.oracle_scan_varlen.argtypes = [P] * 12 + [I] * 5
    lib.oracle_scan_varlen.restype = I
    lib.oracle_state_update_indexed.argtypes = [P, P, I] + [P] * 9 + [I] * 4
    lib.oracle_state_update_indexed.restype = I
    lib.oracle_causal_conv1d.argtypes = [P] * 6 + [I] * 5
    lib.oracle_causal_conv1d.restype = I
    lib.oracle_causal_conv1d_update.argtypes = [P] * 5 + [I] * 4
    lib.oracle_causal_conv1d_update.restype = I
    lib.oracle_scan_bwd.argtypes = [P] * 20 + [I] * 6
    lib.oracle_scan_bwd.restype = I
    lib.oracle_ssd.argtypes = [P] * 11 + [I] * 7
    lib.oracle_ssd.restype = I


class _use_library:
    """Temporarily route this module's calls to another build of the oracle
    source (the mutation tests compile deliberately broken copies)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        lib.oracle_scan.argtypes = self.saved.oracle_scan.argtypes
        lib.oracle_scan.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = self.saved.oracle_state_update.argtypes
        lib.oracle_state_update.restype = ctypes.c_int
        _set_conv_types(lib)
        _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _f64(x, shape=None):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def scan(u, delta, A, B, C, z=None, Dskip=None, dt_bias=None, h0=None, *,
         return_final_state=False, nthreads=None):
    """Selective scan over whole sequences, in fp64.

    u, delta, z: [batch, dim, L]; A: [dim, N]; B, C: [batch, G, N, L];
    Dskip, dt_bias: [dim]; h0: [batch, dim, N].  Returns y [batch, dim, L]
    (and h_final [batch, dim, N] when ``return_final_state``).
    """
    u = _f64(u)
    if u.ndim != 3:
        raise ValueError("u must be [batch, dim, L]")
    batch, dim, L = u.shape
    delta = _f64(delta, u.shape)
    z = _f64(z, u.shape)
    A = _f64(A)
    if A.ndim != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    B = _f64(B)
    if B.ndim != 4 or B.shape[0] != batch or B.shape[2:] != (N, L):
        raise ValueError("B must be [batch, G, N, L]")
    G = B.shape[1]
    C = _f64(C, B.shape)
    Dskip = _f64(Dskip, (dim,))
    dt_bias = _f64(dt_bias, (dim,))
    h0 = _f64(h0, (batch, dim, N))
    y = np.empty((batch, dim, L), dtype=np.float64)
    hf = np.empty((batch, dim, N), dtype=np.float64) if return_final_state else None
    rc = _load().oracle_scan(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(Dskip), _ptr(dt_bias), _ptr(h0), _ptr(y), _ptr(hf),
                             batch, dim, N, L, G, nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_scan rejected its arguments (code {rc})")
    return (y, hf) if return_final_state else y


def state_update(state, u, delta, A, B, C, z=None, Dskip=None, dt_bias=None):
    """One decode step in fp64.  Returns (new_state, y); the input is not modified.

    state: [batch, dim, N]; u, delta, z: [batch, dim]; B, C: [batch, G, N].
    """
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    batch, dim, N = st.shape
    u = _f64(u, (batch, dim))
    delta = _f64(delta, (batch, dim))
    z = _f64(z, (batch, dim))
    A = _f64(A, (dim, N))
    B = _f64(B)
    if B.ndim != 3 or B.shape[0] != batch or B.shape[2] != N:
        raise ValueError("B must be [batch, G, N]")
    G = B.shape[1]
    C = _f64(C, B.shape)
    Dskip = _f64(Dskip, (dim,))
    dt_bias = _f64(dt_bias, (dim,))
    y = np.empty((batch, dim), dtype=np.float64)
    rc = _load().oracle_state_update(_ptr(st), _ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(Dskip), _ptr(dt_bias), _ptr(y),
                                     batch, dim, N, G)
    if rc != 0:
        raise ValueError(f"oracle_state_update rejected its arguments (code {rc})")
    return st, y


def causal_conv1d(x, w, bias=None, x_prev=None, *, silu=True, return_last=False):
    """Short causal depthwise convolution (+ silu) in fp64, the step in front
    of the scan.  x: [batch, dim, L]; w: [dim, W]; bias: [dim]; x_prev:
    [batch, dim, W-1] (the inputs before the sequence, oldest first).
    Returns out [batch, dim, L] (and the last W-1 inputs when ``return_last``)."""
    x = _f64(x)
    if x.ndim != 3:
        raise ValueError("x must be [batch, dim, L]")
    batch, dim, L = x.shape
    w = _f64(w)
    if w.ndim != 2 or w.shape[0] != dim:
        raise ValueError("w must be [dim, W]")
    W = w.shape[1]
    bias = _f64(bias, (dim,))
    x_prev = _f64(x_prev, (batch, dim, W - 1))
    out = np.empty((batch, dim, L), dtype=np.float64)
    last = np.empty((batch, dim, W - 1), dtype=np.float64) if return_last else None
    rc = _load().oracle_causal_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev), _ptr(out), _ptr(last),
                                      batch, dim, L, W, int(bool(silu)))
    if rc != 0:
        raise ValueError(f"oracle_causal_conv1d rejected its arguments (code {rc})")
    return (out, last) if return_last else out


def causal_conv1d_update(conv_state, x, w, bias=None, *, silu=True):
    """One decode token of the convolution in fp64.  Returns (new_state, out);
    the input state is not modified.  conv_state: [batch, dim, W-1]; x: [batch, dim]."""
    x = _f64(x)
    batch, dim = x.shape
    w = _f64(w)
    if w.ndim != 2 or w.shape[0] != dim:
        raise ValueError("w must be [dim, W]")
    W = w.shape[1]
    st = np.array(conv_state, dtype=np.float64, copy=True, order="C").reshape(batch, dim, W - 1)
    bias = _f64(bias, (dim,))
    out = np.empty((batch, dim), dtype=np.float64)
    rc = _load().oracle_causal_conv1d_update(_ptr(st) if W > 1 else None, _ptr(x), _ptr(w), _ptr(bias),
                                             _ptr(out), batch, dim, W, int(bool(silu)))
    if rc != 0:
        raise ValueError(f"oracle_causal_conv1d_update rejected its arguments (code {rc})")
    return st, out


def scan_varlen(u, delta, A, B, C, cu_seqlens, z=None, Dskip=None, dt_bias=None, h0=None, *,
                return_final_state=False):
    """Packed variable-length scan in fp64: sequence s occupies times
    [cu_seqlens[s], cu_seqlens[s+1]) of one row and starts from h0[s] (or 0).
    u, delta, z: [dim, T]; B, C: [G, N, T]; h0: [nseq, dim, N].  Returns y
    [dim, T] (and h_final [nseq, dim, N] when ``return_final_state``)."""
    u = _f64(u)
    if u.ndim != 2:
        raise ValueError("u must be [dim, T]")
    dim, T = u.shape
    delta = _f64(delta, u.shape)
    z = _f64(z, u.shape)
    A = _f64(A)
    if A.ndim != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    B = _f64(B)
    if B.ndim != 3 or B.shape[1:] != (N, T):
        raise ValueError("B must be [G, N, T]")
    G = B.shape[0]
    C = _f64(C, B.shape)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    nseq = cu.size - 1
    Dskip = _f64(Dskip, (dim,))
    dt_bias = _f64(dt_bias, (dim,))
    h0 = _f64(h0, (nseq, dim, N))
    y = np.empty((dim, T), dtype=np.float64)
    hf = np.empty((nseq, dim, N), dtype=np.float64) if return_final_state else None
    rc = _load().oracle_scan_varlen(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                                    _ptr(dt_bias), _ptr(h0), _ptr(cu), _ptr(y), _ptr(hf), dim, N, T, G, nseq)
    if rc != 0:
        raise ValueError(f"oracle_scan_varlen rejected its arguments (code {rc})")
    return (y, hf) if return_final_state else y


def state_update_indexed(state_pool, state_indices, u, delta, A, B, C, z=None, Dskip=None, dt_bias=None):
    """One decode step on a pool of states in fp64: row b advances slot
    state_indices[b] (negative: padding, untouched, y row left as NaN).
    Returns (new_pool, y); the input pool is not modified."""
    pool = np.array(state_pool, dtype=np.float64, copy=True, order="C")
    nslots, dim, N = pool.shape
    idx = np.ascontiguousarray(np.asarray(state_indices, dtype=np.int32))
    batch = idx.size
    u = _f64(u, (batch, dim))
    delta = _f64(delta, (batch, dim))
    z = _f64(z, (batch, dim))
    A = _f64(A, (dim, N))
    B = _f64(B)
    if B.ndim != 3 or B.shape[0] != batch or B.shape[2] != N:
        raise ValueError("B must be [batch, G, N]")
    G = B.shape[1]
    C = _f64(C, B.shape)
    Dskip = _f64(Dskip, (dim,))
    dt_bias = _f64(dt_bias, (dim,))
    y = np.full((batch, dim), np.nan, dtype=np.float64)
    rc = _load().oracle_state_update_indexed(_ptr(pool), _ptr(idx), nslots, _ptr(u), _ptr(delta), _ptr(z),
                                             _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip), _ptr(dt_bias), _ptr(y),
                                             batch, dim, N, G)
    if rc != 0:
        raise ValueError(f"oracle_state_update_indexed rejected its arguments (code {rc})")
    return pool, y



def scan_bwd(u, delta, A, B, C, dy, z=None, Dskip=None, dt_bias=None, h0=None, dh_final=None, *,
             nthreads=None):
    """Gradients of the selective scan in fp64, given dy = dLoss/dy [batch,
    dim, L] and optionally dh_final = dLoss/dh_final [batch, dim, N].

    Returns a dict with du, ddelta, dz (None without z) [batch, dim, L]; dA
    [dim, N]; dB, dC [batch, G, N, L]; dD, ddt_bias [dim]; dh0 [batch, dim, N]
    (the gradient with respect to the initial state, zero or not)."""
    u = _f64(u)
    if u.ndim != 3:
        raise ValueError("u must be [batch, dim, L]")
    batch, dim, L = u.shape
    delta = _f64(delta, u.shape)
    z = _f64(z, u.shape)
    dy = _f64(dy, u.shape)
    A = _f64(A)
    if A.ndim != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    B = _f64(B)
    if B.ndim != 4 or B.shape[0] != batch or B.shape[2:] != (N, L):
        raise ValueError("B must be [batch, G, N, L]")
    G = B.shape[1]
    C = _f64(C, B.shape)
    Dskip = _f64(Dskip, (dim,))
    dt_bias = _f64(dt_bias, (dim,))
    h0 = _f64(h0, (batch, dim, N))
    dh_final = _f64(dh_final, (batch, dim, N))
    out = dict(du=np.empty(u.shape), ddelta=np.empty(u.shape), dz=np.empty(u.shape) if z is not None else None,
               dA=np.empty((dim, N)), dB=np.empty(B.shape), dC=np.empty(B.shape), dD=np.empty(dim),
               ddt_bias=np.empty(dim), dh0=np.empty((batch, dim, N)))
    rc = _load().oracle_scan_bwd(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                                 _ptr(dt_bias), _ptr(h0), _ptr(dy), _ptr(dh_final),
                                 _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dz"]), _ptr(out["dA"]),
                                 _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["ddt_bias"]),
                                 _ptr(out["dh0"]), batch, dim, N, L, G, nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_scan_bwd rejected its arguments (code {rc})")
    return out


def ssd(x, delta, A, B, C, z=None, Dskip=None, dt_bias=None, h0=None, *, headdim,
        return_final_state=False, nthreads=None):
    """SSD (Mamba-2) layer over whole sequences, in fp64: the recurrence with a
    scalar decay A[h], step delta[b, h, t] and skip Dskip[h] per head.

    x, z: [batch, nheads * headdim, L]; delta: [batch, nheads, L]; A, Dskip,
    dt_bias: [nheads]; B, C: [batch, G, N, L]; h0: [batch, nheads * headdim, N].
    Returns y [batch, nheads * headdim, L] (and h_final when asked).
    """
    x = _f64(x)
    if x.ndim != 3:
        raise ValueError("x must be [batch, nheads * headdim, L]")
    batch, dim, L = x.shape
    if dim % headdim != 0:
        raise ValueError("the channel count must be a multiple of headdim")
    nheads = dim // headdim
    delta = _f64(delta, (batch, nheads, L))
    z = _f64(z, x.shape)
    A = _f64(A, (nheads,))
    B = _f64(B)
    if B.ndim != 4 or B.shape[0] != batch or B.shape[3] != L:
        raise ValueError("B must be [batch, G, N, L]")
    G, N = B.shape[1], B.shape[2]
    C = _f64(C, B.shape)
    Dskip = _f64(Dskip, (nheads,))
    dt_bias = _f64(dt_bias, (nheads,))
    h0 = _f64(h0, (batch, dim, N))
    y = np.empty((batch, dim, L), dtype=np.float64)
    hf = np.empty((batch, dim, N), dtype=np.float64) if return_final_state else None
    rc = _load().oracle_ssd(_ptr(x), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                            _ptr(dt_bias), _ptr(h0), _ptr(y), _ptr(hf),
                            batch, nheads, headdim, N, L, G, nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_ssd rejected its arguments (code {rc})")
    return (y, hf) if return_final_state else y
