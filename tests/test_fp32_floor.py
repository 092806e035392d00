"""Pins the reading of the fp32 max-rel tolerance, on the CPU.

The fp32 I/O tolerance is rel-L2 <= 1e-5 and max relative error <= 1e-4
against the fp64 oracle; it does not say what an element near zero is
measured relative to.  The tests read it as
max_i |y_i - r_i| / max(|r_i|, 1e-2 * rms(r)).  These tests show why the
guard cannot be tighter: a correctly rounded fp32 evaluation of the
recurrence (``tests/fp32_model.py``: each operation rounded once, exp and
log correctly rounded -- the best that fp32 arithmetic can do on this
sequence of operations) already scores above 1e-4 on the fp32 workload
itself (batch 1, 64 channels, N 16, L 256, unit recipe, seed 0) once the
guard is 1e-3 * rms, while it stays far inside 1e-4 with 1e-2 * rms, and its
rel-L2 stays two orders below 1e-5.  Outputs near zero come from
cancellation among the 16 terms of C.h (eightmm.github.io "Mamba", Main
Claim: y = C h), whose fp32 rounding floor is about 1e-7 of the terms, not of
their sum.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_109_b300 import inputs as I

from fp32_model import scan_fp32
from parity import F32_MAX_REL, F32_REL_L2, MAX_REL_GUARD, max_rel, rel_l2


def _ideal_fp32(shape, recipe, seed):
    x = I.make_scan_inputs(*shape, io="f32", recipe=recipe, seed=seed)
    f = x.as_f64()
    ref = oracle.scan(**f)
    got = scan_fp32(f["u"], f["delta"], f["A"], f["B"], f["C"], z=f["z"], Dskip=f["Dskip"],
                    dt_bias=f["dt_bias"])
    return got, ref


def test_fp32_model_is_fp32_accurate():
    """The model itself: its state after a short scan matches the oracle to
    a few fp32 ulps (so it is an fp32 evaluation, not a broken one)."""
    x = I.make_scan_inputs(1, 8, 16, 40, 1, io="f32", recipe="scaled", seed=3, with_h0=True)
    f = x.as_f64()
    ry, rh = oracle.scan(**f, return_final_state=True)
    gy, gh = scan_fp32(f["u"], f["delta"], f["A"], f["B"], f["C"], z=f["z"], Dskip=f["Dskip"],
                       dt_bias=f["dt_bias"], h0=f["h0"], return_final_state=True)
    assert rel_l2(gh, rh) < 1e-6
    assert rel_l2(gy, ry) < 1e-6
    assert gy.dtype == np.float32


def test_tight_guard_fails_for_ideal_fp32_on_the_fp32_workload():
    """batch 1, 64 channels, N 16, L 256, fp32, unit recipe, seed 0: the
    ideal fp32 evaluation exceeds 1e-4 under a 1e-3 * rms guard."""
    got, ref = _ideal_fp32((1, 64, 16, 256, 1), "unit", 0)
    assert rel_l2(got, ref) < F32_REL_L2 / 50
    assert max_rel(got, ref, guard=1e-3) > F32_MAX_REL
    assert max_rel(got, ref, guard=MAX_REL_GUARD) < F32_MAX_REL / 5


@pytest.mark.parametrize("shape,recipe,seed", [
    ((2, 128, 16, 512, 1), "unit", 1),
    ((1, 64, 16, 1024, 1), "unit", 0),
])
def test_tight_guard_fails_on_longer_unit_inputs(shape, recipe, seed):
    """The same holds on larger inputs of the unit recipe (B, C ~ N(0, 1):
    the most cancellation in C.h), and the 1e-2 * rms guard keeps a margin
    of at least 2x for the ideal fp32 evaluation."""
    got, ref = _ideal_fp32(shape, recipe, seed)
    assert max_rel(got, ref, guard=1e-3) > F32_MAX_REL
    assert max_rel(got, ref, guard=MAX_REL_GUARD) < F32_MAX_REL / 2


def test_guard_matches_the_parity_tests():
    assert MAX_REL_GUARD == 1e-2


def test_ideal_fp32_on_the_summary_lane_test_input():
    """The input of the GPU test of the summary pass's lane split (batch 2,
    150 channels, N 16, L 480, scaled recipe, seed 36, with h0, drawn on the
    CPU): the ideal fp32 evaluation meets the full fp32 tolerance (max-rel
    about 0.6 of it: an element just above the guard with heavy cancellation),
    so the GPU test holds that input to the full tolerance too."""
    x = I.make_scan_inputs(2, 150, 16, 480, 1, io="f32", recipe="scaled", seed=36, with_h0=True)
    f = x.as_f64()
    ref = oracle.scan(**f)
    got = scan_fp32(f["u"], f["delta"], f["A"], f["B"], f["C"], z=f["z"], Dskip=f["Dskip"],
                    dt_bias=f["dt_bias"], h0=f["h0"])
    assert rel_l2(got, ref) < F32_REL_L2 / 50
    assert max_rel(got, ref) < F32_MAX_REL
