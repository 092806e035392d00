"""The SSD (Mamba-2) layer on the tensor cores against the fp64 SSD oracle
(itself pinned to the selective-scan oracle and the quadratic duality form),
on identical seeded inputs.  The tensor-core contractions take bf16 operands,
so every case is held to the bf16 tolerance (rel-L2 <= 5e-3) and the final
state to the state tolerance.  Shapes span several chunks, a ragged tail, two
groups, no gate, an initial state, and the full workload."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_REL_L2, STATE_REL_L2, rel_l2, to_np
from selective_state_space_109_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    from selective_state_space_109_b300 import ssm as m
    return m


def run(ssm, x, headdim=64, **kw):
    return ssm.ssd_fwd(x["x"], x["delta"], x["A"], x["B"], x["C"], z=x["z"], D=x["D"], dt_bias=x["dt_bias"],
                       h0=x["h0"], headdim=headdim, return_final_state=True, **kw)


def ref(x, headdim=64):
    f = lambda t: None if t is None else to_np(t)
    return oracle.ssd(f(x["x"]), f(x["delta"]), f(x["A"]), f(x["B"]), f(x["C"]), z=f(x["z"]), Dskip=f(x["D"]),
                      dt_bias=f(x["dt_bias"]), h0=f(x["h0"]), headdim=headdim, return_final_state=True)


@pytest.mark.parametrize("batch,nheads,L,G,with_z,with_h0", [
    (1, 2, 128, 1, True, False),     # one chunk
    (1, 2, 512, 1, True, True),      # several chunks, carried state, initial state
    (2, 4, 392, 2, True, True),      # ragged last chunk, two groups
    (1, 3, 200, 1, False, False),    # no gate, ragged
    (1, 1, 8, 1, True, True),        # shorter than a chunk
])
def test_ssd_matches_oracle(ssm, batch, nheads, L, G, with_z, with_h0):
    x = I.make_ssd_inputs(batch, nheads, 64, 128, L, G, seed=80 + L, device="cuda", with_z=with_z,
                          with_h0=with_h0)
    y, hf = run(ssm, x)
    torch.cuda.synchronize()
    ry, rh = ref(x)
    e, eh = rel_l2(to_np(y), ry), rel_l2(to_np(hf), rh)
    print(f"L={L}: y rel_l2 {e:.2e}, h_final rel_l2 {eh:.2e}")
    assert e <= BF16_REL_L2, f"y rel_l2 {e:.3e}"
    assert eh <= STATE_REL_L2, f"h_final rel_l2 {eh:.3e}"
    assert ssm.device_status() == 0


@pytest.mark.parametrize("N", [16, 32, 64])
def test_ssd_smaller_state_sizes(ssm, N):
    """State sizes below 128 run on the 128-state tiles, the rows past N
    loaded as zeros: several chunks, a ragged last one, two groups, an
    initial state and its final state."""
    x = I.make_ssd_inputs(2, 4, 64, N, 392, 2, seed=70 + N, device="cuda", with_h0=True)
    y, hf = run(ssm, x)
    torch.cuda.synchronize()
    ry, rh = ref(x)
    e, eh = rel_l2(to_np(y), ry), rel_l2(to_np(hf), rh)
    print(f"N={N}: y rel_l2 {e:.2e}, h_final rel_l2 {eh:.2e}")
    assert e <= BF16_REL_L2, f"y rel_l2 {e:.3e}"
    assert eh <= STATE_REL_L2, f"h_final rel_l2 {eh:.3e}"
    assert ssm.device_status() == 0


def test_ssd_empty_sequence_copies_h0(ssm):
    x = I.make_ssd_inputs(1, 2, 64, 128, 0, seed=90, device="cuda", with_h0=True)
    y, hf = run(ssm, x)
    torch.cuda.synchronize()
    assert torch.equal(hf, x["h0"])


def test_ssd_rejects_unsupported_shapes(ssm):
    x = I.make_ssd_inputs(1, 2, 32, 128, 64, seed=91, device="cuda")
    with pytest.raises(ssm.SsmError):
        run(ssm, x, headdim=32)


def test_ssd_full_workload_sampled_heads(ssm):
    """The measured workload (batch 2, 64 heads of 64 channels, N 128, L 2048)
    at full size on the GPU; 16 heads compared with the oracle in full."""
    w = I.WORKLOADS["ssd_bf16_b2_h64_p64_n128_l2048"]
    x = I.make_ssd_inputs(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["seqlen"], w["ngroups"], seed=0,
                          device="cuda")
    y, hf = run(ssm, x)
    torch.cuda.synchronize()
    P = w["headdim"]
    heads = [0, 1, 17, 31, 32, 47, 62, 63]
    for b in range(w["batch"]):
        for h in heads:
            sub = {k: v for k, v in x.items()}
            sub["x"] = x["x"][b:b + 1, h * P:(h + 1) * P]
            sub["z"] = x["z"][b:b + 1, h * P:(h + 1) * P]
            sub["delta"] = x["delta"][b:b + 1, h:h + 1]
            sub["A"], sub["D"], sub["dt_bias"] = x["A"][h:h + 1], x["D"][h:h + 1], x["dt_bias"][h:h + 1]
            sub["B"], sub["C"] = x["B"][b:b + 1], x["C"][b:b + 1]
            ry, rh = ref(sub)
            e = rel_l2(to_np(y[b:b + 1, h * P:(h + 1) * P]), ry)
            eh = rel_l2(to_np(hf[b:b + 1, h * P:(h + 1) * P]), rh)
            assert e <= BF16_REL_L2, f"b={b} h={h}: y rel_l2 {e:.3e}"
            assert eh <= STATE_REL_L2, f"b={b} h={h}: h_final rel_l2 {eh:.3e}"


def test_ssd_writes_exactly_its_outputs(ssm):
    """Canary: y and the final state are views into larger buffers filled with
    a sentinel (a ragged last chunk, two groups); the kernel must write exactly
    their elements."""
    x = I.make_ssd_inputs(1, 4, 64, 128, 200, 2, seed=93, device="cuda", with_h0=True)
    n, m = x["x"].numel(), x["h0"].numel()
    big_y = torch.full((n + 8192,), 7.0, dtype=torch.bfloat16, device="cuda")
    big_h = torch.full((m + 8192,), 7.0, dtype=torch.float32, device="cuda")
    y = big_y[4096:4096 + n].view_as(x["x"])
    hf = big_h[4096:4096 + m].view_as(x["h0"])
    run(ssm, x, out=y, h_final=hf)
    torch.cuda.synchronize()
    assert torch.all(big_y[:4096] == 7.0) and torch.all(big_y[4096 + n:] == 7.0)
    assert torch.all(big_h[:4096] == 7.0) and torch.all(big_h[4096 + m:] == 7.0)
    ry, rh = ref(x)
    assert rel_l2(to_np(y), ry) <= BF16_REL_L2
    assert rel_l2(to_np(hf), rh) <= STATE_REL_L2
