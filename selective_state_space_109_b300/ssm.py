"""Python binding of libssmscan.so (the C ABI in include/ssm_scan.h).

Argument marshalling only: shapes and dtypes are checked, outputs are
allocated with torch on the inputs' device, and the C entry point is called
with raw device pointers on the current torch CUDA stream.  Every step of the
computation runs in the library's CUDA kernels.  Importing this module loads
the library and raises ImportError if it is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssmscan.so")

SSM_F32 = 0
SSM_BF16 = 1
STATUS_NAMES = {0: "SSM_OK", 1: "SSM_ERR_INVALID_ARG", 2: "SSM_ERR_UNSUPPORTED",
                3: "SSM_ERR_MISALIGNED", 4: "SSM_ERR_WORKSPACE_TOO_SMALL",
                5: "SSM_ERR_TIMEOUT", 6: "SSM_ERR_CUDA"}


class SsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES.get(status, f"status {status}")
        extra = ""
        if status == 6:
            extra = f" (cudaError {lib.ssm_last_cuda_error()})"
        super().__init__(f"{where}: {name}{extra}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m selective_state_space_109_b300.build` "
            "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.ssm_abi_version.argtypes = []
    L.ssm_abi_version.restype = I
    L.ssm_status_string.argtypes = [I]
    L.ssm_status_string.restype = ctypes.c_char_p
    L.ssm_last_cuda_error.argtypes = []
    L.ssm_last_cuda_error.restype = I
    L.ssm_scan_fwd.argtypes = [P] * 9 + [I] * 6 + [P]
    L.ssm_scan_fwd.restype = I
    L.ssm_scan_fwd_chunked_workspace_size.argtypes = [I] * 6
    L.ssm_scan_fwd_chunked_workspace_size.restype = Z
    L.ssm_scan_fwd_chunked.argtypes = [P] * 11 + [I] * 6 + [P, Z, P]
    L.ssm_scan_fwd_chunked.restype = I
    L.ssm_workspace_status.argtypes = [P, Z, P]
    L.ssm_workspace_status.restype = I
    L.ssm_scan_fwd_chunked_static.argtypes = [P] * 11 + [I] * 6 + [P]
    L.ssm_scan_fwd_chunked_static.restype = I
    L.ssm_scan_plan.argtypes = [I] * 7 + [P] * 4
    L.ssm_scan_plan.restype = I
    L.ssm_device_status.argtypes = [I, P]
    L.ssm_device_status.restype = I
    L.ssm_set_pass_timer.argtypes = [P, P]
    L.ssm_set_pass_timer.restype = I
    L.ssm_state_update.argtypes = [P] * 10 + [I] * 5 + [P]
    L.ssm_state_update.restype = I
    L.ssm_scan_fwd_varlen.argtypes = [P] * 12 + [I] * 6 + [P]
    L.ssm_scan_fwd_varlen.restype = I
    L.ssm_state_update_pooled.argtypes = [P, P, I] + [P] * 9 + [I] * 5 + [P]
    L.ssm_state_update_pooled.restype = I
    L.ssm_causal_conv1d_fwd.argtypes = [P] * 6 + [I] * 6 + [P]
    L.ssm_causal_conv1d_fwd.restype = I
    L.ssm_causal_conv1d_update.argtypes = [P] * 5 + [I] * 5 + [P]
    L.ssm_causal_conv1d_update.restype = I
    L.ssm_scan_bwd_workspace_size.argtypes = [I] * 6
    L.ssm_scan_bwd_workspace_size.restype = Z
    L.ssm_scan_bwd.argtypes = [P] * 20 + [I] * 6 + [P, Z, P]
    L.ssm_scan_bwd.restype = I
    L.ssm_ssd_fwd.argtypes = [P] * 11 + [I] * 7 + [P]
    L.ssm_ssd_fwd.restype = I
    D = ctypes.POINTER(ctypes.c_double)
    L.ssm_probe_alu_rates.argtypes = [P, D, D, D, P]
    L.ssm_probe_alu_rates.restype = I
    return L


lib = _load()


def _io_code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return SSM_F32
    if dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported I/O dtype {dtype} (float32 or bfloat16)")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scan_shapes(u, A, B):
    if u.dim() != 3 or A.dim() != 2 or B.dim() != 4:
        raise ValueError("expected u [batch, dim, L], A [dim, N], B [batch, G, N, L]")
    batch, dim, L = u.shape
    N = A.shape[1]
    G = B.shape[1]
    return batch, dim, N, L, G


def _validate_scan(u, delta, z, A, B, C, D, dt_bias):
    if u.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    batch, dim, N, L, G = _scan_shapes(u, A, B)
    dev, io = u.device, u.dtype
    _io_code(io)
    _check(u, "u", (batch, dim, L), io, dev)
    _check(delta, "delta", (batch, dim, L), io, dev)
    _check(z, "z", (batch, dim, L), io, dev)
    _check(A, "A", (dim, N), torch.float32, dev)
    _check(B, "B", (batch, G, N, L), io, dev)
    _check(C, "C", (batch, G, N, L), io, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(dt_bias, "dt_bias", (dim,), torch.float32, dev)
    return batch, dim, N, L, G


def scan_fwd(u, delta, A, B, C, z=None, D=None, dt_bias=None, *, out=None) -> torch.Tensor:
    """y = selective scan of (u, delta, A, B, C) with skip D and gate silu(z); h0 = 0."""
    batch, dim, N, L, G = _validate_scan(u, delta, z, A, B, C, D, dt_bias)
    y = torch.empty_like(u) if out is None else out
    _check(y, "out", u.shape, u.dtype, u.device)
    with torch.cuda.device(u.device):
        st = lib.ssm_scan_fwd(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                              _ptr(dt_bias), _ptr(y), batch, dim, N, L, G, _io_code(u.dtype),
                              _stream_handle(u.device))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd")
    return y


def scan_plan(batch, dim, dstate, seqlen, ngroups, dtype, chunked=True) -> dict:
    """The library's launch plan for this problem: lanes per channel, time
    chunks, kernels per call and whether the TMA-staged kernels run."""
    vals = [ctypes.c_int(0) for _ in range(4)]
    st = lib.ssm_scan_plan(batch, dim, dstate, seqlen, ngroups, _io_code(dtype), int(bool(chunked)),
                           *[ctypes.byref(v) for v in vals])
    if st != 0:
        raise SsmError(st, "ssm_scan_plan")
    return dict(lanes=vals[0].value, chunks=vals[1].value, kernels=vals[2].value, staged=bool(vals[3].value))


def chunked_workspace_size(batch, dim, dstate, seqlen, ngroups, dtype) -> int:
    return int(lib.ssm_scan_fwd_chunked_workspace_size(batch, dim, dstate, seqlen, ngroups,
                                                       _io_code(dtype)))


def alloc_workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    return torch.empty(int(nbytes), dtype=torch.uint8, device=device)


def scan_fwd_chunked(u, delta, A, B, C, z=None, D=None, dt_bias=None, h0=None, *, out=None,
                     h_final=None, workspace=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Selective scan from initial state h0 (zeros if None); returns (y, h_final)."""
    batch, dim, N, L, G = _validate_scan(u, delta, z, A, B, C, D, dt_bias)
    _check(h0, "h0", (batch, dim, N), torch.float32, u.device)
    y = torch.empty_like(u) if out is None else out
    _check(y, "out", u.shape, u.dtype, u.device)
    hf = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device) if h_final is None else h_final
    _check(hf, "h_final", (batch, dim, N), torch.float32, u.device)
    need = chunked_workspace_size(batch, dim, N, L, G, u.dtype)
    ws = alloc_workspace(need, u.device) if workspace is None else workspace
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    with torch.cuda.device(u.device):
        st = lib.ssm_scan_fwd_chunked(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C),
                                      _ptr(D), _ptr(dt_bias), _ptr(h0), _ptr(y), _ptr(hf),
                                      batch, dim, N, L, G, _io_code(u.dtype), _ptr(ws), ws_bytes,
                                      _stream_handle(u.device))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_chunked")
    return y, hf


def workspace_status(workspace: torch.Tensor) -> int:
    """Synchronises the current stream and returns the device-side status code."""
    with torch.cuda.device(workspace.device):
        return int(lib.ssm_workspace_status(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream_handle(workspace.device)))


def device_status(clear: bool = False, device=None) -> int:
    """Synchronises the current stream and returns the library's device error
    status (0 = no bounded device-side wait has given up)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib.ssm_device_status(int(bool(clear)), _stream_handle(dev)))


def set_pass_timer(begin=None, end=None) -> None:
    """Registers two torch.cuda.Event objects (enable_timing=True) that later
    forward scan calls from this thread record around the launch of their
    fused pass; set_pass_timer() clears the hook."""
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None
    st = lib.ssm_set_pass_timer(b, e)
    if st != 0:
        raise SsmError(st, "ssm_set_pass_timer")


def ssd_fwd(x, delta, A, B, C, z=None, D=None, dt_bias=None, h0=None, *, headdim, out=None, h_final=None,
            return_final_state=False):
    """SSD (Mamba-2) layer: x, z [batch, nheads * headdim, L] bf16; delta
    [batch, nheads, L] bf16; A, D, dt_bias [nheads] fp32; B, C [batch, G, N, L]
    bf16; h0 [batch, nheads * headdim, N] fp32.  Returns y (and h_final)."""
    if x.device.type != "cuda" or x.dim() != 3 or B.dim() != 4:
        raise ValueError("expected CUDA tensors x [batch, dim, L], B [batch, G, N, L]")
    batch, dim, L = x.shape
    if dim % headdim != 0:
        raise ValueError("the channel count must be a multiple of headdim")
    nheads = dim // headdim
    G, N = B.shape[1], B.shape[2]
    dev, io = x.device, x.dtype
    _check(x, "x", (batch, dim, L), io, dev)
    _check(delta, "delta", (batch, nheads, L), io, dev)
    _check(z, "z", (batch, dim, L), io, dev)
    _check(A, "A", (nheads,), torch.float32, dev)
    _check(B, "B", (batch, G, N, L), io, dev)
    _check(C, "C", (batch, G, N, L), io, dev)
    _check(D, "D", (nheads,), torch.float32, dev)
    _check(dt_bias, "dt_bias", (nheads,), torch.float32, dev)
    _check(h0, "h0", (batch, dim, N), torch.float32, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", x.shape, io, dev)
    hf = h_final
    if return_final_state and hf is None:
        hf = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    _check(hf, "h_final", (batch, dim, N), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_ssd_fwd(_ptr(x), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                             _ptr(h0), _ptr(y), _ptr(hf), batch, nheads, headdim, N, L, G, _io_code(io),
                             _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_ssd_fwd")
    return (y, hf) if (return_final_state or h_final is not None) else y


def probe_alu_rates(device=None) -> dict:
    """MUFU.EX2 results and fp32 FMAs per SM per nanosecond on the device (see
    ssm_probe_alu_rates in the C header); synchronises."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    ex2, ffma, mix = ctypes.c_double(0.0), ctypes.c_double(0.0), ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        st = lib.ssm_probe_alu_rates(_ptr(sink), ctypes.byref(ex2), ctypes.byref(ffma), ctypes.byref(mix),
                                     _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_probe_alu_rates")
    return dict(ex2_per_sm_ns=ex2.value, ffma_per_sm_ns=ffma.value, mix_updates_per_sm_ns=mix.value)


def state_update(state, u, delta, A, B, C, z=None, D=None, dt_bias=None, *, out=None,
                 state_indices=None) -> torch.Tensor:
    """One decode step: updates ``state`` [batch, dim, N] in place, returns y
    [batch, dim].  With ``state_indices`` ([batch] int32), ``state`` is a pool
    [nslots, dim, N] and row b advances slot state_indices[b] (outside
    [0, nslots): a padding row, whose y is left unwritten)."""
    if state.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if state.dim() != 3 or B.dim() != 3:
        raise ValueError("expected state [batch, dim, N], B [batch, G, N]")
    nslots, dim, N = state.shape
    batch = u.shape[0]
    G = B.shape[1]
    dev, io = state.device, u.dtype
    _io_code(io)
    if state_indices is None and nslots != batch:
        raise ValueError("state must be [batch, dim, N] without state_indices")
    _check(state, "state", (nslots, dim, N), torch.float32, dev)
    _check(state_indices, "state_indices", (batch,), torch.int32, dev)
    _check(u, "u", (batch, dim), io, dev)
    _check(delta, "delta", (batch, dim), io, dev)
    _check(z, "z", (batch, dim), io, dev)
    _check(A, "A", (dim, N), torch.float32, dev)
    _check(B, "B", (batch, G, N), io, dev)
    _check(C, "C", (batch, G, N), io, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(dt_bias, "dt_bias", (dim,), torch.float32, dev)
    y = torch.empty((batch, dim), dtype=io, device=dev) if out is None else out
    _check(y, "out", (batch, dim), io, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_state_update_pooled(_ptr(state), _ptr(state_indices), nslots, _ptr(u), _ptr(delta), _ptr(z),
                                         _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias), _ptr(y), batch, dim, N,
                                         G, _io_code(io), _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_state_update_pooled")
    return y


def causal_conv1d(x, w, bias=None, x_prev=None, *, silu=True, out=None, x_last=None) -> torch.Tensor:
    """The short causal depthwise convolution in front of the scan:
    out[b,d,l] = silu(bias[d] + sum_k w[d,k] x[b,d,l-(W-1)+k]), with x_prev
    [batch, dim, W-1] as the inputs before the sequence (zeros if None).
    x: [batch, dim, L] (float32 or bfloat16); w: [dim, W] float32, W <= 4.
    ``x_last`` (optional, [batch, dim, W-1]) receives the next segment's history."""
    if x.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if x.dim() != 3 or w.dim() != 2:
        raise ValueError("expected x [batch, dim, L], w [dim, W]")
    batch, dim, L = x.shape
    W = w.shape[1]
    dev, io = x.device, x.dtype
    _io_code(io)
    _check(x, "x", (batch, dim, L), io, dev)
    _check(w, "w", (dim, W), torch.float32, dev)
    _check(bias, "bias", (dim,), torch.float32, dev)
    _check(x_prev, "x_prev", (batch, dim, W - 1), io, dev)
    _check(x_last, "x_last", (batch, dim, W - 1), io, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", x.shape, io, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_causal_conv1d_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev), _ptr(y), _ptr(x_last),
                                       batch, dim, L, W, int(bool(silu)), _io_code(io), _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_causal_conv1d_fwd")
    return y


def causal_conv1d_update(conv_state, x, w, bias=None, *, silu=True, out=None) -> torch.Tensor:
    """One decode token of the convolution: conv_state [batch, dim, W-1] (the
    last W-1 inputs, oldest first) is advanced in place; returns out [batch, dim]."""
    if x.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if x.dim() != 2 or w.dim() != 2:
        raise ValueError("expected x [batch, dim], w [dim, W]")
    batch, dim = x.shape
    W = w.shape[1]
    dev, io = x.device, x.dtype
    _io_code(io)
    _check(conv_state, "conv_state", (batch, dim, W - 1), io, dev)
    _check(w, "w", (dim, W), torch.float32, dev)
    _check(bias, "bias", (dim,), torch.float32, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", x.shape, io, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_causal_conv1d_update(_ptr(conv_state), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), batch, dim,
                                          W, int(bool(silu)), _io_code(io), _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_causal_conv1d_update")
    return y


def scan_fwd_varlen(u, delta, A, B, C, cu_seqlens, z=None, D=None, dt_bias=None, h0=None, *,
                    out=None, h_final=None, return_final_state=False):
    """Scan of a packed batch: u, delta, z [dim, T]; B, C [G, N, T];
    cu_seqlens [nseq + 1] int32 (device); h0, h_final [nseq, dim, N].
    Sequence s occupies times [cu_seqlens[s], cu_seqlens[s+1]) and starts
    from h0[s] (or 0).  Returns y (and h_final when ``return_final_state``)."""
    if u.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if u.dim() != 2 or A.dim() != 2 or B.dim() != 3 or cu_seqlens.dim() != 1:
        raise ValueError("expected u [dim, T], A [dim, N], B [G, N, T], cu_seqlens [nseq + 1]")
    dim, T = u.shape
    N = A.shape[1]
    G = B.shape[0]
    nseq = cu_seqlens.shape[0] - 1
    dev, io = u.device, u.dtype
    _io_code(io)
    for t, name, shape, dt in ((u, "u", (dim, T), io), (delta, "delta", (dim, T), io), (z, "z", (dim, T), io),
                               (A, "A", (dim, N), torch.float32), (B, "B", (G, N, T), io),
                               (C, "C", (G, N, T), io), (D, "D", (dim,), torch.float32),
                               (dt_bias, "dt_bias", (dim,), torch.float32), (h0, "h0", (nseq, dim, N), torch.float32),
                               (cu_seqlens, "cu_seqlens", (nseq + 1,), torch.int32)):
        _check(t, name, shape, dt, dev)
    y = torch.empty_like(u) if out is None else out
    _check(y, "out", u.shape, io, dev)
    hf = h_final
    if hf is None and return_final_state:
        hf = torch.empty((nseq, dim, N), dtype=torch.float32, device=dev)
    _check(hf, "h_final", (nseq, dim, N), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_scan_fwd_varlen(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(dt_bias), _ptr(h0), _ptr(cu_seqlens), _ptr(y), _ptr(hf), dim, N, T, G,
                                     nseq, _io_code(io), _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_varlen")
    return (y, hf) if return_final_state else y



def bwd_workspace_size(batch, dim, dstate, seqlen, ngroups, dtype) -> int:
    return int(lib.ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, ngroups, _io_code(dtype)))


def scan_bwd(u, delta, A, B, C, dy, z=None, D=None, dt_bias=None, h0=None, dh_final=None, *,
             want_dh0=True, out=None, workspace=None) -> dict:
    """Gradients of the selective scan given dy = dLoss/dy [batch, dim, L]
    (and dh_final = dLoss/dh_final [batch, dim, N], or None).

    Returns a dict: du, ddelta, dz (None without z) [batch, dim, L] in the
    I/O type; dA [dim, N], dB and dC [batch, G, N, L], dD and ddt_bias [dim]
    (None when D / dt_bias is None), dh0 [batch, dim, N] (None unless
    want_dh0) in fp32.  ``out`` may hold preallocated tensors under the same
    keys."""
    batch, dim, N, L, G = _validate_scan(u, delta, z, A, B, C, D, dt_bias)
    dev, io = u.device, u.dtype
    _check(dy, "dy", (batch, dim, L), io, dev)
    _check(h0, "h0", (batch, dim, N), torch.float32, dev)
    _check(dh_final, "dh_final", (batch, dim, N), torch.float32, dev)
    o = dict(out or {})
    f32 = torch.float32
    specs = dict(du=((batch, dim, L), io, True), ddelta=((batch, dim, L), io, True),
                 dz=((batch, dim, L), io, z is not None), dA=((dim, N), f32, True),
                 dB=((batch, G, N, L), f32, True), dC=((batch, G, N, L), f32, True),
                 dD=((dim,), f32, D is not None), ddt_bias=((dim,), f32, dt_bias is not None),
                 dh0=((batch, dim, N), f32, bool(want_dh0)))
    for k, (shape, dt, wanted) in specs.items():
        if not wanted:
            o[k] = None
            continue
        if o.get(k) is None:
            o[k] = torch.empty(shape, dtype=dt, device=dev)
        _check(o[k], k, shape, dt, dev)
    need = bwd_workspace_size(batch, dim, N, L, G, io)
    ws = alloc_workspace(need, dev) if workspace is None else workspace
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    with torch.cuda.device(dev):
        st = lib.ssm_scan_bwd(_ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                              _ptr(h0), _ptr(dy), _ptr(dh_final), _ptr(o["du"]), _ptr(o["ddelta"]), _ptr(o["dz"]),
                              _ptr(o["dA"]), _ptr(o["dB"]), _ptr(o["dC"]), _ptr(o["dD"]), _ptr(o["ddt_bias"]),
                              _ptr(o["dh0"]), batch, dim, N, L, G, _io_code(io), _ptr(ws), ws_bytes,
                              _stream_handle(dev))
    if st != 0:
        raise SsmError(st, "ssm_scan_bwd")
    return o


class SelectiveScanFn(torch.autograd.Function):
    """The scan as a differentiable torch op: forward ``scan_fwd_chunked``,
    backward ``scan_bwd`` (no states stored between the two; the backward
    recomputes them).  Gradients arrive in each input's dtype (dB, dC are
    accumulated in fp32 and cast)."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, z, D, dt_bias, h0):
        y, hf = scan_fwd_chunked(u, delta, A, B, C, z=z, D=D, dt_bias=dt_bias, h0=h0)
        ctx.save_for_backward(u, delta, A, B, C, z, D, dt_bias, h0)
        return y, hf

    @staticmethod
    def backward(ctx, dy, dhf):
        u, delta, A, B, C, z, D, dt_bias, h0 = ctx.saved_tensors
        dy = torch.zeros_like(u) if dy is None else dy.to(u.dtype).contiguous()
        dhf = None if dhf is None else dhf.float().contiguous()
        g = scan_bwd(u, delta, A, B, C, dy, z=z, D=D, dt_bias=dt_bias, h0=h0, dh_final=dhf,
                     want_dh0=h0 is not None and ctx.needs_input_grad[8])
        cast = lambda t, like: None if t is None else t.to(like.dtype)
        return (g["du"], g["ddelta"], g["dA"], cast(g["dB"], B), cast(g["dC"], C), g["dz"], g["dD"],
                g["ddt_bias"], g["dh0"])


def selective_scan(u, delta, A, B, C, z=None, D=None, dt_bias=None, h0=None):
    """Differentiable selective scan: returns (y, h_final); torch autograd
    calls this library's backward pass."""
    return SelectiveScanFn.apply(u, delta, A, B, C, z, D, dt_bias, h0)
