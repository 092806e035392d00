"""The pins must be able to fail: each mutant below is the oracle source with
one plausible slip planted in it (compiled here, on the CPU).  For every
mutant at least one of the oracle pins (scan, convolution, packed batches,
backward pass, SSD) has to raise."""
import os
import subprocess

import pytest

import oracle
import test_oracle_bwd_pins as bwd_pins
import test_oracle_conv_pins as conv_pins
import test_oracle_varlen_pins as varlen_pins
import test_oracle_pins as pins
import test_oracle_ssd_pins as ssd_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTANTS = {
    "skip_term_dropped": ("double yt = acc + dskip * ut;", "double yt = acc;"),
    "bias_after_softplus": ("softplus(J->delta[row + t] + bias)", "(softplus(J->delta[row + t]) + bias)"),
    "decay_sign_flipped": ("exp(dt * J->A[(size_t)d * N + n])", "exp(-dt * J->A[(size_t)d * N + n])"),
    "readout_uses_B": ("acc += J->C[bc + (size_t)n * L + t] * h[n];", "acc += J->B[bc + (size_t)n * L + t] * h[n];"),
    "readout_before_update": (
        "h[n] = abar * h[n] + bx;\n            acc += J->C[bc + (size_t)n * L + t] * h[n];",
        "acc += J->C[bc + (size_t)n * L + t] * h[n];\n            h[n] = abar * h[n] + bx;"),
    "gate_skips_the_skip_path": ("if (J->z) yt *= silu(J->z[row + t]);",
                                 "if (J->z) yt = acc * silu(J->z[row + t]) + dskip * ut;"),
    "h0_ignored": ("h[n] = J->h0 ? J->h0[((size_t)b * J->dim + d) * N + n] : 0.0;", "h[n] = 0.0;"),
    "group_index_interleaved": ("const int g = d / (J->dim / J->ngroups);\n    const size_t row",
                                "const int g = d % J->ngroups;\n    const size_t row"),
    "B_one_step_late": ("const double bx = dt * J->B[bc + (size_t)n * L + t] * ut;",
                        "const double bx = dt * J->B[bc + (size_t)n * L + (t > 0 ? t - 1 : 0)] * ut;"),
    "softplus_without_abs": ("log1p(exp(-fabs(x)))", "log1p(exp(-x))"),
    "input_term_without_step": ("const double bx = dt * J->B[", "const double bx = J->B["),
    "decode_gate_dropped": ("if (z) yt *= silu(z[bd]);", ""),
    # the short convolution in front of the scan
    "conv_taps_reversed": ("acc += w[(size_t)d * W + k] * conv_input(x, x_prev, row, prow, W, l - (W - 1) + k);",
                           "acc += w[(size_t)d * W + (W - 1 - k)] * conv_input(x, x_prev, row, prow, W, l - (W - 1) + k);"),
    "conv_window_one_step_late": ("conv_input(x, x_prev, row, prow, W, l - (W - 1) + k);",
                                  "conv_input(x, x_prev, row, prow, W, l - W + k);"),
    "conv_history_ignored": ("return x_prev ? x_prev[prow + (size_t)((W - 1) + t)] : 0.0;", "return 0.0;"),
    "conv_history_reversed": ("x_prev[prow + (size_t)((W - 1) + t)]", "x_prev[prow + (size_t)(-1 - t)]"),
    "conv_bias_dropped": ("                double acc = bias ? bias[d] : 0.0;\n                for (int k = 0; k < W; k++)",
                          "                double acc = 0.0;\n                for (int k = 0; k < W; k++)"),
    "conv_silu_dropped": ("out[row + (size_t)l] = silu_act ? silu(acc) : acc;", "out[row + (size_t)l] = acc;"),
    "conv_state_shift_reversed": ("for (int k = 0; k + 1 < W - 1; k++) st[k] = st[k + 1];",
                                  "for (int k = W - 2; k > 0; k--) st[k] = st[k - 1];"),
    "conv_update_newest_tap_wrong": ("acc += w[(size_t)d * W + (W - 1)] * x[bd];", "acc += w[(size_t)d * W] * x[bd];"),
    # packed variable-length batches and the pooled decode step
    "varlen_no_reset_between_sequences": (
        "            for (int n = 0; n < N; n++)\n                h[n] = h0 ? h0[((size_t)s * dim + d) * N + n] : 0.0;",
        "            for (int n = 0; n < N; n++)\n                if (s == 0) h[n] = h0 ? h0[((size_t)s * dim + d) * N + n] : 0.0;"),
    "varlen_first_sequence_h0_for_all": ("h[n] = h0 ? h0[((size_t)s * dim + d) * N + n] : 0.0;",
                                         "h[n] = h0 ? h0[((size_t)0 * dim + d) * N + n] : 0.0;"),
    "varlen_group_interleaved": ("const size_t bc = (size_t)g * (size_t)N * (size_t)T;",
                                 "const size_t bc = (size_t)(d % ngroups) * (size_t)N * (size_t)T;"),
    "pooled_decode_reads_batch_row": ("double *h = &state_pool[((size_t)slot * dim + d) * N];",
                                      "double *h = &state_pool[((size_t)b * dim + d) * N];"),
    # the backward pass
    "bwd_dB_without_step": ("J->dB[k] += l * dt * ut;", "J->dB[k] += l * ut;"),
    "bwd_adjoint_not_decayed": ("lam[n] = abar * l;", "lam[n] = l;"),
    "bwd_dDelta_drops_decay_term": ("ddelta_t += l * (J->B[k] * ut + Ad[n] * abar * hprev[n]);",
                                    "ddelta_t += l * J->B[k] * ut;"),
    "bwd_dC_uses_previous_state": ("J->dC[k] += gt * hcur[n];", "J->dC[k] += gt * hprev[n];"),
    "bwd_dz_drops_silu_derivative_term": ("sg * (1.0 + zt * (1.0 - sg))", "sg"),
    "bwd_softplus_derivative_without_bias": ("ddelta_t * sigmoid(J->delta[row + t] + bias)",
                                             "ddelta_t * sigmoid(J->delta[row + t])"),
    "bwd_du_skip_dropped": ("J->du[row + t] = gt * dskip + dt * dsum_b;", "J->du[row + t] = dt * dsum_b;"),
    "bwd_dA_uses_current_state": ("J->dA[(size_t)d * N + n] += l * dt * abar * hprev[n];",
                                  "J->dA[(size_t)d * N + n] += l * dt * abar * hcur[n];"),
    "bwd_dh_final_ignored": ("lam[n] = J->dhf ? J->dhf[st + n] : 0.0;", "lam[n] = 0.0;"),
    "bwd_worker_sums_overwritten": ("dA[i] += J->dA[i];", "dA[i] = J->dA[i];"),
    # the SSD (Mamba-2) layer
    "ssd_head_group_interleaved": ("const int g = h / (J->nheads / J->ngroups);",
                                   "const int g = h % J->ngroups;"),
    "ssd_decay_per_channel_index": ("const double a = J->A[h];", "const double a = J->A[0];"),
    "ssd_input_without_step": ("*hp = abar * *hp + dt * J->B[bc + (size_t)n * L + t] * xt;",
                               "*hp = abar * *hp + J->B[bc + (size_t)n * L + t] * xt;"),
    "ssd_readout_uses_B": ("acc += J->C[bc + (size_t)n * L + t] * *hp;", "acc += J->B[bc + (size_t)n * L + t] * *hp;"),
    "ssd_skip_dropped": ("double yt = acc + dskip * xt;", "double yt = acc;"),
}

PIN_TESTS = [
    lambda: pins.test_hand_worked_golden_cases(),
    lambda: pins.test_single_step_closed_form(False),
    lambda: pins.test_single_step_closed_form(True),
    lambda: pins.test_geometric_series_n1_constant_inputs(),
    lambda: pins.test_matches_causal_matrix_mixer(True, True),
    lambda: pins.test_groups_read_their_own_B_C(),
    lambda: pins.test_time_invariant_case_is_a_convolution(),
    lambda: pins.test_vanishing_step_leaves_only_skip_path(),
    lambda: pins.test_large_step_overwrites_state(),
    lambda: pins.test_decode_steps_equal_one_scan(),
    lambda: pins.test_decode_single_step_from_zero_state(),
    lambda: conv_pins.test_conv_hand_worked_golden(),
    lambda: conv_pins.test_conv_matches_numpy_convolve(4, True, True),
    lambda: conv_pins.test_conv_impulse_response(),
    lambda: conv_pins.test_conv_history_splits_sequence(9),
    lambda: conv_pins.test_conv_decode_steps_equal_conv(),
    lambda: conv_pins.test_conv_width_one_is_pointwise(),
    lambda: varlen_pins.test_varlen_equals_each_sequence_alone(),
    lambda: varlen_pins.test_pooled_decode_equals_gathered_decode(),
    lambda: bwd_pins.test_gradients_match_finite_differences(True, True, 2),
    lambda: bwd_pins.test_single_step_closed_form(True),
    lambda: bwd_pins.test_empty_sequence_passes_dh_final_to_h0(),
    lambda: bwd_pins.test_threads_do_not_change_sums(),
    lambda: ssd_pins.test_ssd_equals_the_scan_with_spread_parameters(2, True),
    lambda: ssd_pins.test_ssd_equals_the_quadratic_duality_form(2),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(mutated), "-lm"], check=True)
    failures = 0
    with oracle._use_library(str(lib)):
        for pin in PIN_TESTS:
            try:
                pin()
            except AssertionError:
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"
