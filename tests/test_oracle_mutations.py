"""The oracle's pins must catch plausible mistakes.

Each case compiles a copy of oracle/gdn_oracle.c with one planted mistake
(on the CPU, into a temporary directory), points the oracle wrappers at it
and runs the pin tests that should catch it; at least one must fail.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_cursor_protocol as cp
from tests import test_oracle_derived_d_pins as dd
from tests import test_oracle_pins as pins
from tests import test_oracle_prefill_pins as pp
from tests import test_oracle_snapshot_pins as sp

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTATIONS = {
    "sign_of_delta": ("double d = beta * (v[i] - u);", "double d = beta * (u - v[i]);"),
    "decay_after_delta": (
        "    /* decay first, then the delta against the decayed state ([blog] §12.1) */\n"
        "    if (per_key_gate) {",
        "    if (0) {"),
    "q_not_normalised": ("orc_l2norm(K, q_raw, eps, qh);",
                         "for (int j = 0; j < K; ++j) qh[j] = q_raw[j];"),
    "ring_ignores_base": ("return (base + o) & (L - 1);", "return o & (L - 1);"),
    "gqa_head_map": ("const int h = hv / (HV / H);\n    double *o_row0",
                     "const int h = hv % H;\n    double *o_row0"),
    "margin_T_not_2T": ("(wp + 2 * d->T > d->L)", "(wp + d->T > d->L)"),
    "fold_keeps_base": ("cur->cache_base[slot] = ring_pos(base, wp, d->L);",
                        "cur->cache_base[slot] = base;"),
    "softplus_threshold": ("return x > 20.0 ? x : log1p(exp(x));",
                           "return x > 2.0 ? x : log1p(exp(x));"),
    "history_off_by_one": ("for (int o = 0; o < W; ++o) {", "for (int o = 1; o < W; ++o) {"),
    "kda_gate_scalar": ("for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= exp(g[j]);",
                        "for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= exp(g[0]);"),
    "prefill_keeps_base": (
        "        if (!prefill_row_ok(d, cur, slot, from_zero, &st)) continue;\n"
        "        cur->write_pos[slot] = 0;\n"
        "        cur->cache_base[slot] = 0;\n",
        "        if (!prefill_row_ok(d, cur, slot, from_zero, &st)) continue;\n"
        "        cur->write_pos[slot] = 0;\n"),
    "prefill_ignores_from_zero": ("if (J->from_zero) memset(S, 0, sizeof(double) * (size_t)V * K);",
                                  "(void)0;"),
    "prefill_reads_out_before_step": (
        "        orc_step(V, K, d->per_key_gate, S, J->v + (tok * HV + hv) * V, J->k + (tok * H + h) * K, g,\n"
        "                 beta, d->l2_eps);\n"
        "        orc_readout(V, K, S, J->q + (tok * H + h) * K, d->l2_eps, d->scale, J->out + (tok * HV + hv) * V);\n",
        "        orc_readout(V, K, S, J->q + (tok * H + h) * K, d->l2_eps, d->scale, J->out + (tok * HV + hv) * V);\n"
        "        orc_step(V, K, d->per_key_gate, S, J->v + (tok * HV + hv) * V, J->k + (tok * H + h) * K, g,\n"
        "                 beta, d->l2_eps);\n"),
    "window_d_without_state": ("if (d_out) d_out[i] = d;", "if (d_out) d_out[i] = beta * v[i];"),
    "snapshot_commits_last_draft": ("snap + (((size_t)bb * T + acc - 1) * HV + hv) * VK",
                                    "snap + (((size_t)bb * T + T - 1) * HV + hv) * VK"),
    "snapshot_stores_state_before_step": (
        "                orc_step(V, K, d->per_key_gate, S, v + (tok * HV + hv) * V, k + (tok * H + h) * K, g,\n"
        "                         orc_gate_beta(b[tok * HV + hv]), d->l2_eps);\n"
        "                orc_readout(V, K, S, q + (tok * H + h) * K, d->l2_eps, d->scale, out + (tok * HV + hv) * V);\n"
        "                memcpy(snap + (tok * HV + hv) * VK, S, sizeof(double) * VK);\n",
        "                memcpy(snap + (tok * HV + hv) * VK, S, sizeof(double) * VK);\n"
        "                orc_step(V, K, d->per_key_gate, S, v + (tok * HV + hv) * V, k + (tok * H + h) * K, g,\n"
        "                         orc_gate_beta(b[tok * HV + hv]), d->l2_eps);\n"
        "                orc_readout(V, K, S, q + (tok * H + h) * K, d->l2_eps, d->scale, out + (tok * HV + hv) * V);\n"),
}

CHECKS = [
    pins.test_gate_special_values,
    pins.test_gate_against_library_routines,
    pins.test_readout_normalises_q,
    lambda: pins.test_step_equals_dense_gdn_formula(3, 5),
    lambda: pins.test_step_equals_dense_kda_formula(3, 5),
    lambda: pins.test_verify_equals_closed_form_ut_transform(False, 5),
    lambda: pins.test_verify_equals_closed_form_ut_transform(True, 5),
    pins.test_fold_then_verify_equals_verify_with_history_bitwise,
    lambda: cp.test_oracle_cursors_follow_protocol_b(16, 4),
    cp.test_golden_ring_walk_l8,
    cp.test_golden_margin_rule,
    lambda: pp.test_prefill_equals_dense_recurrence(False, True),
    lambda: pp.test_prefill_equals_dense_recurrence(True, False),
    pp.test_prefill_in_two_calls_equals_one_call_bitwise,
    pp.test_prefill_status_padding_and_unfolded_rows,
    lambda: sp.test_snapshot_verify_equals_dense_recurrence(False),
    sp.test_snapshot_commit_copies_the_accepted_state,
    sp.test_snapshot_and_ring_agree_on_outputs_and_committed_state,
    lambda: dd.test_window_d_equals_closed_form_and_rank_one_identity(True, 3),
    lambda: dd.test_state_reconstructed_from_checkpoint_and_deltas(False),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "gdn_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-pthread", str(mutated),
                    "-o", str(so), "-lm"], check=True)
    failures = 0
    try:
        oracle.use_library(str(so))
        for check in CHECKS:
            try:
                check()
            except AssertionError:
                failures += 1
    finally:
        oracle.use_library(None)
    assert failures > 0, f"no pin caught the planted mistake {name}"
