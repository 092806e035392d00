"""ssm_scan_fwd_chunked_static: the chunked scan for callers that cannot
allocate device memory (for example a plugin whose host runtime owns every
device buffer and passes only inputs and outputs, or a decode loop that must
not call cudaMalloc/cudaFree because they can wait on in-flight GPU work).  Its
scratch is a fixed library-owned array, so the GPU test checks that two calls
in a row through the C ABI give what the workspace entry point gives, and
what the fp64 oracle gives.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

from parity import (BF16_REL_L2, F32_REL_L2, STATE_REL_L2, assert_close, oracle_compare_blocks, oracle_scan,
                    rel_l2, to_np)
from selective_state_space_109_b300 import inputs as I

STATIC_SCRATCH_BYTES = 16 * 1024 * 1024


def _lib():
    from selective_state_space_109_b300 import ssm
    return ssm


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(ssm, x, y, hf, h0=None):
    batch, dim, L = x.u.shape
    N, G = x.A.shape[1], x.B.shape[1]
    io = 0 if x.u.dtype == torch.float32 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ssm.lib.ssm_scan_fwd_chunked_static(
        _ptr(x.u), _ptr(x.delta), _ptr(x.z), _ptr(x.A), _ptr(x.B), _ptr(x.C), _ptr(x.D),
        _ptr(x.dt_bias), _ptr(h0), _ptr(y), _ptr(hf), batch, dim, N, L, G, io, stream)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice(monkeypatch):
    ssm = _lib()
    # Two different problems back to back, each split into four time chunks
    # (forced, and checked through the plan query), so the carry runs through
    # the static array and the second call reuses the array the first filled.
    monkeypatch.setenv("SSM_FORCE_CHUNKS", "4")
    cases = [dict(batch=2, dim=128, dstate=16, seqlen=2048, ngroups=1, io="bf16", seed=41, h0=False),
             dict(batch=1, dim=96, dstate=16, seqlen=1000, ngroups=2, io="f32", seed=42, h0=True)]
    for c in cases:
        dt = torch.float32 if c["io"] == "f32" else torch.bfloat16
        plan = ssm.scan_plan(c["batch"], c["dim"], c["dstate"], c["seqlen"], c["ngroups"], dt)
        assert plan["chunks"] == 4, plan
        x = I.make_scan_inputs(c["batch"], c["dim"], c["dstate"], c["seqlen"], c["ngroups"], io=c["io"],
                               recipe="scaled", seed=c["seed"], device="cuda", with_h0=c["h0"])
        h0 = x.h0 if c["h0"] else None
        y_ref, h_ref = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias,
                                            h0=h0)
        y = torch.full_like(x.u, float("nan"))
        hf = torch.full((c["batch"], c["dim"], c["dstate"]), float("nan"), device="cuda")
        assert _call_static(ssm, x, y, hf, h0) == 0
        torch.cuda.synchronize()
        tol = F32_REL_L2 if c["io"] == "f32" else BF16_REL_L2
        assert rel_l2(to_np(y), to_np(y_ref)) <= tol
        assert rel_l2(to_np(hf), to_np(h_ref)) <= STATE_REL_L2
        # ... and the static call's own result against the fp64 oracle.
        ref_y, ref_h = oracle_scan(x, h0=h0, final_state=True)
        assert_close(to_np(y), ref_y, c["io"], "static entry point")
        assert rel_l2(to_np(hf), ref_h) <= STATE_REL_L2
    assert ssm.device_status() == 0


def test_static_entry_checks_arguments_before_enqueuing():
    """Argument checks only (fake pointers; each call returns before anything
    is enqueued): a misaligned input, a missing output, bad sizes."""
    ssm = _lib()
    P, Q = 0x10000, 0x10008
    f = ssm.lib.ssm_scan_fwd_chunked_static
    assert f(Q, P, P, P, P, P, P, P, None, P, P, 2, 64, 16, 256, 1, 1, None) == 3  # SSM_ERR_MISALIGNED
    assert f(P, P, P, P, P, P, P, P, None, None, P, 2, 64, 16, 256, 1, 1, None) == 1  # no y
    assert f(P, P, P, P, P, P, P, P, None, P, P, 2, 64, 16, 256, 3, 1, None) == 1  # dim % ngroups
    assert f(P, P, P, P, P, P, P, P, None, P, P, 2, 64, 12, 256, 1, 1, None) == 2  # dstate 12


@pytest.mark.gpu
def test_static_scratch_caps_the_chunk_count(monkeypatch):
    """8 x 2048 channels with 16 time chunks forced: the summaries of 15 chunks
    (15 MiB x 2) do not fit the array, so the call plans the 8 chunks whose 7
    summaries do, and must still agree with the workspace entry point."""
    ssm = _lib()
    monkeypatch.setenv("SSM_FORCE_CHUNKS", "16")
    x = I.make_scan_inputs(8, 2048, 16, 512, 1, io="bf16", recipe="scaled", seed=43, device="cuda",
                           with_h0=True)
    per_chunk = 8 * 2048 * 2 * 16 * 4
    assert 256 + 7 * per_chunk <= STATIC_SCRATCH_BYTES < 256 + 8 * per_chunk
    y_ref, h_ref = ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, h0=x.h0)
    y = torch.full_like(x.u, float("nan"))
    hf = torch.full((8, 2048, 16), float("nan"), device="cuda")
    assert _call_static(ssm, x, y, hf, x.h0) == 0
    torch.cuda.synchronize()
    assert rel_l2(to_np(y), to_np(y_ref)) <= BF16_REL_L2
    assert rel_l2(to_np(hf), to_np(h_ref)) <= STATE_REL_L2
    e, eh, _ = oracle_compare_blocks(x, y, hf)
    assert e <= BF16_REL_L2 and eh <= STATE_REL_L2, (e, eh)
    assert ssm.device_status() == 0
