"""Seeded synthetic inputs for the selective scan and the decode update.

This module only draws random numbers and lays them out; it holds none of the
scan's arithmetic.  Both the CUDA path (tests, benchmark) and the fp64 oracle
(tests, CPU baseline) take their inputs from here, so the two sides always see
identical values.

Recipes (one per workload family):

* ``"unit"``  -- u, z, delta ~ N(0,1); B, C ~ N(0,1); Dskip = 1;
  dt_bias = softplus^-1(dt) with dt log-uniform on [1e-3, 1e-1];
  A[d, n] = -(n + 1).
* ``"scaled"`` -- as ``"unit"`` but B, C ~ N(0,1)/sqrt(N) and
  Dskip ~ N(1, 0.1) (0.1 read as the standard deviation).

Every tensor draws from its own torch generator, keyed by (seed, tensor name,
decode step), so adding or dropping one tensor never shifts another.  Values
are drawn in fp32 and rounded to bf16 (round-to-nearest-even, torch's
``.to(torch.bfloat16)``) when the I/O type is bf16; A, Dskip, dt_bias and the
decode state always stay fp32.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_TENSOR_IDS = {"u": 1, "delta": 2, "z": 3, "B": 4, "C": 5, "D": 6, "dt": 7,
               "h0": 8, "state": 9, "A": 10, "conv_x": 11, "conv_w": 12, "conv_bias": 13,
               "conv_prev": 14}


def _subseed(seed: int, name: str, step: int = 0) -> int:
    key = f"{seed}/{_TENSOR_IDS[name]}/{step}".encode()
    return int.from_bytes(hashlib.sha256(key).digest()[:8], "little") & ((1 << 63) - 1)


def _gen(seed, name, device, step=0):
    g = torch.Generator(device=device)
    g.manual_seed(_subseed(seed, name, step))
    return g


def _randn(shape, seed, name, device, step=0):
    return torch.randn(shape, generator=_gen(seed, name, device, step), device=device,
                       dtype=torch.float32)


def io_torch_dtype(io: str) -> torch.dtype:
    if io == "f32":
        return torch.float32
    if io == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown I/O type {io!r}")


def dt_bias_values(dim: int, seed: int, device="cpu") -> torch.Tensor:
    """dt_bias = softplus^-1(dt), dt = exp(U(ln 1e-3, ln 1e-1)), computed in fp64, stored fp32."""
    g = _gen(seed, "dt", "cpu")
    r = torch.rand(dim, generator=g, dtype=torch.float64)
    dt = torch.exp(math.log(1e-3) + r * (math.log(1e-1) - math.log(1e-3)))
    return torch.log(torch.expm1(dt)).to(torch.float32).to(device)


def a_values(dim: int, dstate: int, device="cpu") -> torch.Tensor:
    """A[d, n] = -(n + 1) for every channel."""
    return (-(torch.arange(dstate, dtype=torch.float32) + 1.0)).repeat(dim, 1).to(device)


def a_values_random(dim: int, dstate: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """A[d, n] = -U(0.5, 16.5), drawn per element: no structure across n."""
    g = _gen(seed, "A", "cpu")
    return (-(0.5 + 16.0 * torch.rand((dim, dstate), generator=g, dtype=torch.float32))).to(device)


@dataclass
class ScanInputs:
    u: torch.Tensor
    delta: torch.Tensor
    z: Optional[torch.Tensor]
    A: torch.Tensor
    B: torch.Tensor
    C: torch.Tensor
    D: torch.Tensor
    dt_bias: torch.Tensor
    h0: Optional[torch.Tensor] = None

    def to(self, device):
        f = lambda t: None if t is None else t.to(device)
        return ScanInputs(f(self.u), f(self.delta), f(self.z), f(self.A), f(self.B),
                          f(self.C), f(self.D), f(self.dt_bias), f(self.h0))

    def as_f64(self):
        """numpy fp64 copies (exact widening of fp32/bf16) for the oracle."""
        f = lambda t: None if t is None else t.detach().to("cpu", torch.float32).double().numpy()
        return dict(u=f(self.u), delta=f(self.delta), z=f(self.z), A=f(self.A), B=f(self.B),
                    C=f(self.C), Dskip=f(self.D), dt_bias=f(self.dt_bias), h0=f(self.h0))


def make_scan_inputs(batch, dim, dstate, seqlen, ngroups=1, io="f32", recipe="unit",
                     seed=0, device="cpu", with_z=True, with_h0=False) -> ScanInputs:
    """Inputs for one selective-scan call in the documented layouts.

    u, delta, z: [batch, dim, seqlen]; A: [dim, dstate]; B, C:
    [batch, ngroups, dstate, seqlen]; D, dt_bias: [dim]; h0: [batch, dim, dstate].
    """
    dt = io_torch_dtype(io)
    act = (batch, dim, seqlen)
    bc = (batch, ngroups, dstate, seqlen)
    bscale = 1.0 if recipe == "unit" else 1.0 / math.sqrt(dstate)
    if recipe not in ("unit", "scaled"):
        raise ValueError(f"unknown recipe {recipe!r}")
    u = _randn(act, seed, "u", device).to(dt)
    delta = _randn(act, seed, "delta", device).to(dt)
    z = _randn(act, seed, "z", device).to(dt) if with_z else None
    B = (_randn(bc, seed, "B", device) * bscale).to(dt)
    C = (_randn(bc, seed, "C", device) * bscale).to(dt)
    if recipe == "unit":
        D = torch.ones(dim, dtype=torch.float32, device=device)
    else:
        D = 1.0 + 0.1 * _randn((dim,), seed, "D", device)
    h0 = _randn((batch, dim, dstate), seed, "h0", device) if with_h0 else None
    return ScanInputs(u, delta, z, a_values(dim, dstate, device), B, C, D,
                      dt_bias_values(dim, seed, device), h0)


def make_decode_state(batch, dim, dstate, seed=0, device="cpu") -> torch.Tensor:
    """fp32 state [batch, dim, dstate] ~ N(0, 1)."""
    return _randn((batch, dim, dstate), seed, "state", device)


def make_decode_token(batch, dim, dstate, step, ngroups=1, io="bf16", recipe="scaled",
                      seed=0, device="cpu", with_z=True) -> dict:
    """One token for every sequence of the batch: u, delta, z [batch, dim];
    B, C [batch, ngroups, dstate].  ``step`` keys the draw."""
    dt = io_torch_dtype(io)
    bscale = 1.0 if recipe == "unit" else 1.0 / math.sqrt(dstate)
    return dict(
        u=_randn((batch, dim), seed, "u", device, step).to(dt),
        delta=_randn((batch, dim), seed, "delta", device, step).to(dt),
        z=_randn((batch, dim), seed, "z", device, step).to(dt) if with_z else None,
        B=(_randn((batch, ngroups, dstate), seed, "B", device, step) * bscale).to(dt),
        C=(_randn((batch, ngroups, dstate), seed, "C", device, step) * bscale).to(dt),
    )


def decode_params(dim, dstate, recipe="scaled", seed=0, device="cpu"):
    """Per-channel parameters of the decode workload: A, D, dt_bias."""
    if recipe == "unit":
        D = torch.ones(dim, dtype=torch.float32, device=device)
    else:
        D = 1.0 + 0.1 * _randn((dim,), seed, "D", device)
    return dict(A=a_values(dim, dstate, device), D=D, dt_bias=dt_bias_values(dim, seed, device))


def make_ssd_inputs(batch, nheads, headdim, dstate, seqlen, ngroups=1, io="bf16", seed=0, device="cpu",
                    with_z=True, with_h0=False) -> dict:
    """Inputs of the SSD (Mamba-2) layer: x, z ~ N(0, 1) [batch, nheads *
    headdim, L]; delta ~ N(0, 1) [batch, nheads, L]; B, C ~ N(0, 1/N) [batch, G,
    N, L] (all in the I/O type); per head A = -U(1, 16) (the A = -(n+1) range of
    the scan workloads as one scalar per head), D ~ N(1, 0.1^2) and dt_bias =
    softplus^-1(dt) with dt log-uniform on [1e-3, 1e-1] (fp32); h0 ~ N(0, 1)."""
    dt = io_torch_dtype(io)
    dim = nheads * headdim
    act = (batch, dim, seqlen)
    bc = (batch, ngroups, dstate, seqlen)
    g = _gen(seed, "A", "cpu", step=11)
    out = dict(
        x=_randn(act, seed, "u", "cpu").to(dt),
        delta=_randn((batch, nheads, seqlen), seed, "delta", "cpu").to(dt),
        z=_randn(act, seed, "z", "cpu").to(dt) if with_z else None,
        A=-(1.0 + 15.0 * torch.rand(nheads, generator=g, dtype=torch.float32)),
        B=(_randn(bc, seed, "B", "cpu") / math.sqrt(dstate)).to(dt),
        C=(_randn(bc, seed, "C", "cpu") / math.sqrt(dstate)).to(dt),
        D=1.0 + 0.1 * _randn((nheads,), seed, "D", "cpu"),
        dt_bias=dt_bias_values(nheads, seed, "cpu"),
        h0=_randn((batch, dim, dstate), seed, "h0", "cpu") if with_h0 else None,
    )
    return {k: (v.contiguous().to(device) if v is not None else None) for k, v in out.items()}


def compulsory_bytes_ssd(batch, nheads, headdim, dstate, seqlen, ngroups, io="bf16") -> int:
    """x, z, y ([batch, nheads * headdim, L] each), delta ([batch, nheads, L])
    and B, C ([batch, G, N, L] each)."""
    s = 4 if io == "f32" else 2
    return (3 * batch * nheads * headdim * seqlen + batch * nheads * seqlen + 2 * batch * ngroups * dstate * seqlen) * s


def flops_ssd_chunked(batch, nheads, headdim, dstate, seqlen, chunk=128) -> int:
    """Dense-contraction FLOPs of the chunked SSD evaluation (2 per multiply-add):
    per chunk and head C B^T (Q x Q over N), the mixer times x (Q x P over Q),
    the chunk state (N x P over Q) and the carried-state readout (Q x P over N)."""
    nch = -(-seqlen // chunk)
    Q, P, N = chunk, headdim, dstate
    return 2 * batch * nheads * nch * (Q * Q * N + Q * P * Q + N * P * Q + Q * P * N)


# Named workloads: the sizes of the five synthetic workloads this library is
# checked and measured on.
def make_conv_inputs(batch, dim, seqlen, width=4, io="bf16", seed=0, device="cpu", with_prev=False):
    """Inputs of the short causal convolution in front of the scan: x
    [batch, dim, L] ~ N(0, 1) in the I/O type (the pre-convolution activation,
    same scale as u); w [dim, W] ~ N(0, 1/W) fp32 (unit gain); bias [dim] ~
    N(0, 0.1^2) fp32; optional history [batch, dim, W-1] ~ N(0, 1)."""
    dt = io_torch_dtype(io)
    x = _randn((batch, dim, seqlen), seed, "conv_x", "cpu").to(dt)
    w = (_randn((dim, width), seed, "conv_w", "cpu") / width ** 0.5).float()
    bias = (0.1 * _randn((dim,), seed, "conv_bias", "cpu")).float()
    prev = _randn((batch, dim, width - 1), seed, "conv_prev", "cpu").to(dt) if with_prev else None
    mv = lambda t: None if t is None else t.to(device)
    return dict(x=mv(x), w=mv(w), bias=mv(bias), x_prev=mv(prev))


def make_varlen_inputs(dim, dstate, lengths, ngroups=1, io="bf16", recipe="scaled", seed=0, device="cpu",
                       with_h0=False, row_multiple=1):
    """A packed batch of sequences of the given lengths laid end to end along
    time: the tensors of make_scan_inputs for one row of T = sum(lengths)
    steps (rounded up to a multiple of row_multiple; the rest is padding) with
    the batch axis dropped (u, delta, z [dim, T]; B, C [G, N, T]), h0
    [nseq, dim, N] when asked, and cu_seqlens [nseq + 1] int32."""
    T = -(-int(sum(lengths)) // row_multiple) * row_multiple
    x = make_scan_inputs(1, dim, dstate, T, ngroups, io=io, recipe=recipe, seed=seed, device="cpu")
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    out = dict(u=x.u[0], delta=x.delta[0], z=x.z[0], A=x.A, B=x.B[0], C=x.C[0], D=x.D, dt_bias=x.dt_bias,
               cu_seqlens=cu)
    if with_h0:
        out["h0"] = _randn((len(lengths), dim, dstate), seed, "h0", "cpu")
    return {k: (v.contiguous().to(device) if v is not None else None) for k, v in out.items()}


def varlen_lengths(n, mean, seed=0):
    """n sequence lengths drawn uniformly from [1, 2 * mean - 1] (a serving
    batch: mixed lengths, no padding), from the seeded stream of tensor "dt"."""
    g = _gen(seed, "dt", "cpu", step=7)
    return [int(v) for v in torch.randint(1, 2 * mean, (n,), generator=g)]


def compulsory_bytes_conv(batch, dim, seqlen, io) -> int:
    """x read and out written once ([batch, dim, L] each)."""
    return 2 * batch * dim * seqlen * (4 if io == "f32" else 2)


WORKLOADS = {
    "scan_f32_tiny": dict(kind="scan", batch=1, dim=64, dstate=16, seqlen=256, ngroups=1,
                          io="f32", recipe="unit"),
    "scan_bf16_b2_d1536_l2048": dict(kind="scan", batch=2, dim=1536, dstate=16, seqlen=2048,
                                     ngroups=1, io="bf16", recipe="unit"),
    "scan_bf16_b8_d2048_l4096": dict(kind="scan", batch=8, dim=2048, dstate=16, seqlen=4096,
                                     ngroups=1, io="bf16", recipe="scaled"),
    "scan_bf16_b1_d5120_l65536_final_state": dict(kind="scan", batch=1, dim=5120, dstate=16,
                                                  seqlen=65536, ngroups=1, io="bf16",
                                                  recipe="scaled", final_state=True),
    # Large state: the b2 d1536 L2048 shape with N = 64, 128 and 256 states per channel.
    "scan_bf16_b2_d1536_l2048_n64": dict(kind="scan", batch=2, dim=1536, dstate=64, seqlen=2048,
                                         ngroups=1, io="bf16", recipe="scaled"),
    "scan_bf16_b2_d1536_l2048_n128": dict(kind="scan", batch=2, dim=1536, dstate=128, seqlen=2048,
                                          ngroups=1, io="bf16", recipe="scaled"),
    "scan_bf16_b2_d1536_l2048_n256": dict(kind="scan", batch=2, dim=1536, dstate=256, seqlen=2048,
                                          ngroups=1, io="bf16", recipe="scaled"),
    "decode_b256_d5120": dict(kind="decode", batch=256, dim=5120, dstate=16, ngroups=1,
                              io="bf16", recipe="scaled", steps=1024),
    # SSD (Mamba-2) layer: 64 heads of 64 channels (4096 channels), N 128, L 2048.
    "ssd_bf16_b2_h64_p64_n128_l2048": dict(kind="ssd", batch=2, nheads=64, headdim=64, dstate=128,
                                           seqlen=2048, ngroups=1, io="bf16"),
}


def compulsory_bytes_scan(batch, dim, dstate, seqlen, ngroups, io) -> int:
    """u, delta, z, y ([batch, dim, L] each) plus B and C ([batch, G, N, L] each)."""
    s = 4 if io == "f32" else 2
    return 4 * batch * dim * seqlen * s + 2 * batch * ngroups * dstate * seqlen * s


def compulsory_bytes_bwd(batch, dim, dstate, seqlen, ngroups, io) -> int:
    """Backward pass: reads u, delta, z, dy ([batch, dim, L] each) and B, C
    ([batch, G, N, L] each); writes du, ddelta, dz in the I/O type and dB, dC
    in fp32."""
    s = 4 if io == "f32" else 2
    act, bc = batch * dim * seqlen, batch * ngroups * dstate * seqlen
    return 7 * act * s + 2 * bc * s + 2 * bc * 4


def compulsory_bytes_decode(batch, dim, dstate) -> int:
    """The fp32 state read plus written once per token."""
    return 2 * batch * dim * dstate * 4
