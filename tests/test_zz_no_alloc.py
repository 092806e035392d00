"""ssm_scan_fwd_chunked_static: the chunked scan for callers that cannot
allocate device memory (for example a plugin whose host runtime owns every
device buffer and passes only inputs and outputs, or a decode loop that must
not call cudaMalloc/cudaFree because they can wait on in-flight GPU work).  Its
scratch is a fixed library-owned array, so the GPU test checks that two calls
in a row through the C ABI give what the workspace entry point gives.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

from parity import BF16_REL_L2, F32_REL_L2, STATE_REL_L2, rel_l2, to_np
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
def test_static_scratch_matches_workspace_entry_point_twice():
    ssm = _lib()
    # Two different problems back to back: both plan several time chunks, so
    # the second call reuses the scratch array the first one filled.
    cases = [dict(batch=2, dim=128, dstate=16, seqlen=2048, ngroups=1, io="bf16", seed=41, h0=False),
             dict(batch=1, dim=96, dstate=16, seqlen=1000, ngroups=2, io="f32", seed=42, h0=True)]
    for c in cases:
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
    assert ssm.device_status() == 0


def test_static_scratch_rejects_problems_beyond_its_size(monkeypatch):
    """Argument check only (fake pointers, nothing is launched): 16 time chunks
    over 8 x 2048 channels need 15 * 16384 * 128 bytes of summaries, more than
    the array holds."""
    ssm = _lib()
    monkeypatch.setenv("SSM_FORCE_CHUNKS", "16")
    P = 0x10000
    st = ssm.lib.ssm_scan_fwd_chunked_static(P, P, P, P, P, P, P, P, None, P, P,
                                             8, 2048, 16, 4096, 1, 1, None)
    assert st == 4  # SSM_ERR_WORKSPACE_TOO_SMALL
