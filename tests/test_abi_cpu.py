"""C-ABI checks that need no GPU: the library loads, exports every function
include/*.h declares, and rejects bad arguments before anything touches the
device (these calls return from the host-side checks; no kernel is launched)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_109_b300 import build
    build.build()
    from selective_state_space_109_b300 import ssm
    return ssm.lib


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["ssm_scan_fwd", "ssm_scan_fwd_chunked", "ssm_scan_fwd_chunked_workspace_size",
                     "ssm_state_update", "ssm_workspace_status", "ssm_status_string",
                     "ssm_abi_version", "ssm_last_cuda_error"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version_and_status_strings(lib):
    assert lib.ssm_abi_version() == 1
    for code, name in [(0, b"SSM_OK"), (1, b"SSM_ERR_INVALID_ARG"), (2, b"SSM_ERR_UNSUPPORTED"),
                       (3, b"SSM_ERR_MISALIGNED"), (4, b"SSM_ERR_WORKSPACE_TOO_SMALL"),
                       (5, b"SSM_ERR_TIMEOUT"), (6, b"SSM_ERR_CUDA")]:
        assert lib.ssm_status_string(code) == name


# Fake, never-dereferenced pointer values: the checks only look at their
# presence and alignment.
P = 0x10000
MIS = 0x10008


def scan(lib, u=P, delta=P, z=None, A=P, B=P, C=P, D=None, bias=None, y=P,
         batch=1, dim=4, N=16, L=8, G=1, io=1):
    return lib.ssm_scan_fwd(u, delta, z, A, B, C, D, bias, y, batch, dim, N, L, G, io, None)


def test_scan_argument_errors(lib):
    assert scan(lib, u=None) == 1
    assert scan(lib, A=None) == 1
    assert scan(lib, y=None) == 1
    assert scan(lib, dim=0) == 1
    assert scan(lib, batch=-1) == 1
    assert scan(lib, L=-5) == 1
    assert scan(lib, dim=6, G=4) == 1          # dim % ngroups
    assert scan(lib, N=12) == 2                # unsupported state size
    assert scan(lib, N=512) == 2               # N up to 256
    assert scan(lib, N=128, L=9, B=MIS) == 3   # N = 128 and 256 pass the checks on unaligned rows too
    assert scan(lib, N=256, L=9, B=MIS) == 3
    assert scan(lib, io=7) == 2
    assert scan(lib, B=MIS) == 3               # misaligned
    assert scan(lib, z=MIS) == 3
    assert scan(lib, batch=0, u=None, y=None) == 0  # empty problem: nothing to do


def test_chunked_workspace_rules(lib):
    need = lib.ssm_scan_fwd_chunked_workspace_size(1, 4, 16, 8, 1, 1)
    assert need >= 0
    assert lib.ssm_scan_fwd_chunked_workspace_size(1, 4, 12, 8, 1, 1) == 0  # invalid -> 0
    if need > 0:
        st = lib.ssm_scan_fwd_chunked(P, P, None, P, P, P, None, None, None, P, P,
                                      1, 4, 16, 8, 1, 1, P, need - 1, None)
        assert st == 4
        st = lib.ssm_scan_fwd_chunked(P, P, None, P, P, P, None, None, None, P, P,
                                      1, 4, 16, 8, 1, 1, None, 0, None)
        assert st == 4
    st = lib.ssm_scan_fwd_chunked(P, P, None, P, P, P, None, None, MIS, P, P,
                                  1, 4, 16, 8, 1, 1, P, need, None)
    assert st == 3  # misaligned h0


def test_state_update_argument_errors(lib):
    def call(state=P, u=P, delta=P, z=None, A=P, B=P, C=P, y=P, batch=2, dim=4, N=16, G=1, io=1):
        return lib.ssm_state_update(state, u, delta, z, A, B, C, None, None, y, batch, dim, N, G, io, None)
    assert call(state=None) == 1
    assert call(y=None) == 1
    assert call(dim=0) == 1
    assert call(dim=6, G=4) == 1
    assert call(N=6) == 2
    assert call(state=MIS) == 3
    assert call(batch=0, state=None) == 0


def test_workspace_status_argument_errors(lib):
    assert lib.ssm_workspace_status(None, 256, None) == 1
    assert lib.ssm_workspace_status(P, 8, None) == 1
    assert lib.ssm_workspace_status(MIS, 256, None) == 3


def test_conv_argument_errors(lib):
    """Argument checks of the short convolution (fake pointers; each call
    returns before anything is enqueued)."""
    Q = 0x20000

    def fwd(x=P, w=P, bias=None, prev=None, out=Q, last=None, batch=2, dim=4, L=16, W=4, io=1):
        return lib.ssm_causal_conv1d_fwd(x, w, bias, prev, out, last, batch, dim, L, W, 1, io, None)
    assert fwd(w=None) == 1
    assert fwd(out=None) == 1
    assert fwd(out=P) == 1                    # out is x
    assert fwd(prev=Q + 0x100, last=Q + 0x100) == 1   # history in and out share a buffer
    assert fwd(dim=0) == 1
    assert fwd(W=5) == 2
    assert fwd(W=0) == 2
    assert fwd(io=7) == 2
    assert fwd(x=MIS) == 3
    assert fwd(batch=0, x=None, out=None) == 0

    def upd(state=P, x=Q, w=Q + 0x100, out=Q + 0x200, W=4, io=1):
        return lib.ssm_causal_conv1d_update(state, x, w, None, out, 2, 4, W, 1, io, None)
    assert upd(state=None) == 1
    assert upd(x=None) == 1
    assert upd(out=Q) == 1                    # out is x
    assert upd(W=5) == 2
    assert upd(state=MIS) == 3


def test_varlen_and_pooled_argument_errors(lib):
    """Argument checks of the packed scan and the pooled decode step (fake
    pointers; each call returns before anything is enqueued)."""
    def varlen(u=P, cu=P, dim=8, N=16, T=64, G=1, nseq=3, io=1):
        return lib.ssm_scan_fwd_varlen(u, P, None, P, P, P, None, None, None, cu, P, None, dim, N, T, G, nseq, io,
                                       None)
    assert varlen(nseq=0) == 1
    assert varlen(cu=None) == 1
    assert varlen(cu=MIS) == 3
    assert varlen(N=12) == 2
    assert varlen(N=128, cu=MIS) == 3         # the packed scan takes N = 128 and 256
    assert varlen(N=256, cu=MIS) == 3
    assert varlen(dim=6, G=4) == 1

    def pooled(idx=None, nslots=2, batch=2):
        return lib.ssm_state_update_pooled(P, idx, nslots, P, P, None, P, P, P, None, None, P, batch, 4, 16, 1, 1,
                                           None)
    assert pooled(idx=None, nslots=3) == 1      # without indices the pool is the batch
    assert pooled(idx=P, nslots=0) == 1
    assert pooled(idx=MIS, nslots=4) == 3


def test_bwd_argument_errors(lib):
    """Argument checks of the backward pass (fake pointers; every call below
    fails its checks and returns before anything is enqueued)."""
    Q = 0x40000

    def bwd(u=P, z=None, D=None, bias=None, dy=Q, du=Q + 0x100, dd=Q + 0x200, dz=None, dA=Q + 0x300, dB=Q + 0x400,
            dC=Q + 0x500, dD=None, db=None, dh0=None, ws=None, ws_bytes=0, batch=1, dim=4, N=16, L=8, G=1, io=1):
        return lib.ssm_scan_bwd(u, P, z, P, P, P, D, bias, None, dy, None, du, dd, dz, dA, dB, dC, dD, db, dh0,
                                batch, dim, N, L, G, io, ws, ws_bytes, None)
    assert bwd(dy=None) == 1
    assert bwd(du=None) == 1
    assert bwd(dB=None) == 1
    assert bwd(dA=None) == 1
    assert bwd(z=P + 0x600, dz=None) == 1          # a gated forward needs dz
    assert bwd(D=P + 0x700, dD=None) == 1          # D given: dD required
    assert bwd(bias=P + 0x800, db=None) == 1       # dt_bias given: ddt_bias required
    assert bwd(du=P) == 1                          # du aliases u
    assert bwd(dim=6, G=4) == 1
    assert bwd(N=12) == 2
    assert bwd(N=512) == 2
    assert bwd(io=9) == 2
    assert bwd(dy=MIS) == 3
    assert bwd(dh0=MIS) == 3
    # 300 steps are three chunks: summaries need a workspace
    need = lib.ssm_scan_bwd_workspace_size(1, 4, 16, 300, 1, 1)
    assert need == 3 * 4 * 16 * 3 * 4
    assert bwd(L=300) == 4
    assert bwd(L=300, ws=Q + 0x900, ws_bytes=need - 16) == 4
    assert lib.ssm_scan_bwd_workspace_size(1, 4, 16, 128, 1, 1) == 0   # one chunk: no workspace
    assert lib.ssm_scan_bwd_workspace_size(2, 4, 64, 129, 1, 1) == 3 * 2 * 4 * 64 * 3 * 4
    # The chunk length fills whole waves of three CTAs on each of 148 SMs: b2
    # d1536 L2048 takes 20 tiles of 8 steps (13 chunks, 96 x 13 CTAs) where
    # 16 tiles would leave a partial fourth wave; b8 d2048 L4096 keeps 16.
    assert lib.ssm_scan_bwd_workspace_size(2, 1536, 16, 2048, 1, 1) == 13 * 2 * 1536 * 16 * 3 * 4
    assert lib.ssm_scan_bwd_workspace_size(8, 2048, 16, 4096, 1, 1) == 32 * 8 * 2048 * 16 * 3 * 4
    assert lib.ssm_scan_bwd_workspace_size(2, 1440, 16, 520, 1, 1) == 4 * 2 * 1440 * 16 * 3 * 4  # 17 tiles
    assert bwd(batch=0, u=None, dy=None, du=None, dd=None, dA=None, dB=None, dC=None) == 0  # empty problem


def ssd(lib, x=P, delta=P, z=None, A=P, B=P, C=P, D=None, bias=None, h0=None, y=P, hf=None,
        batch=1, nheads=2, P_=64, N=128, L=64, G=1, io=1):
    return lib.ssm_ssd_fwd(x, delta, z, A, B, C, D, bias, h0, y, hf, batch, nheads, P_, N, L, G, io, None)


def test_ssd_argument_checks(lib):
    assert ssd(lib, io=0) == 2            # fp32 I/O: the tensor-core path is bf16 only
    assert ssd(lib, P_=32) == 2           # head dimension other than 64
    assert ssd(lib, N=256) == 2           # state size above the 128-state tiles
    assert ssd(lib, N=48) == 2            # state size other than 16, 32, 64, 128
    assert ssd(lib, L=12) == 2            # rows not whole 16-byte packets
    assert ssd(lib, nheads=3, G=2) == 1   # heads do not split into the groups
    assert ssd(lib, nheads=0) == 1
    assert ssd(lib, y=None) == 1          # missing output
    assert ssd(lib, A=None) == 1
    assert ssd(lib, x=MIS) == 3           # misaligned input
    assert ssd(lib, batch=0) == 0         # nothing to do


def test_pass_timer_arguments(lib):
    # Both events or neither: one alone is an argument error (checked on the
    # host; the events are never touched without a GPU).
    fake = ctypes.c_void_p(0x1000)
    assert lib.ssm_set_pass_timer(fake, None) == 1
    assert lib.ssm_set_pass_timer(None, fake) == 1
    assert lib.ssm_set_pass_timer(None, None) == 0
