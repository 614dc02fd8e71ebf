"""Planted mistakes: the oracle's pins must catch every one.

Each case copies oracle/spec_oracle.c, turns one expression into a plausible
mistake (a dropped term, a flipped comparison or sign, a wrong index,
transposed operands, a wrong search order), compiles the copy with gcc, binds
it in place of the oracle's library for the length of the test, and runs pins
that must then fail. A control compiles the unchanged source the same way and
runs every pin named here, which must pass, so a failure can only come from
the planted change.

The mistakes live only in the temporary copy; the oracle's source and the
CUDA library are never touched. None of them can read outside an array, so a
mistake shows as a failed pin, not as a crash. CPU only.
"""
import ctypes
import importlib
import subprocess

import pytest

import oracle

SRC = oracle._SRC

PINS = "test_oracle_pins"
TEMP = "test_oracle_temperature_pins"
TOP_P = "test_oracle_top_p_pins"
IRLS = "test_oracle_irls_pins"
AV = "test_oracle_av_pins"
NGRAM = "test_oracle_ngram_pins"
DEC = "test_oracle_decision_report_pins"

# name: (expression in spec_oracle.c, the planted mistake, pins that catch it
# as (module, test, keyword arguments))
PLANTED = {
    # softmax and row statistics
    "lse_drops_the_max": (
        "    *ok = 1;\n    return m + log(s);\n", "    *ok = 1;\n    return log(s);\n",
        [(PINS, "test_row_stats_against_scipy", {}), (PINS, "test_log_ratio_matches_logsumexp", {})]),
    "entropy_not_normalised": (
        "    return h / log((double)V);", "    return h;",
        [(PINS, "test_entropy_closed_forms", {}), (PINS, "test_row_stats_against_scipy", {})]),
    "entropy_sign": (
        "if (p[v] > 0.0) h -= p[v] * log(p[v]);", "if (p[v] > 0.0) h += p[v] * log(p[v]);",
        [(PINS, "test_entropy_closed_forms", {}), (PINS, "test_row_stats_against_scipy", {})]),
    "feature_sign": (
        "rest > 0.0 ? log(q[amax]) - log(rest) : INFINITY", "rest > 0.0 ? log(rest) - log(q[amax]) : INFINITY",
        [(PINS, "test_logit_qmax_is_capped_at_30", {"gap": 5.0}),
         (PINS, "test_confidence_is_sigmoid_of_affine_feature", {})]),
    "feature_complement_includes_max": (
        "        if (v != amax) rest += q[v];", "        rest += q[v];",
        [(PINS, "test_logit_qmax_clamps_when_complement_vanishes", {}), (PINS, "test_row_stats_against_scipy", {})]),
    "argmax_ties_to_highest": (
        "        if (z > bz) { bz = z; best = v; }", "        if (z >= bz) { bz = z; best = v; }",
        [(PINS, "test_greedy_is_argmax_match_with_ties", {})]),
    "log_ratio_sign": (
        "lr = (zx >= zs_t ? sc * zx - lse_t : -INFINITY) - (qx >= zs_d ? sc * qx - lse_d : -INFINITY);",
        "lr = (qx >= zs_d ? sc * qx - lse_d : -INFINITY) - (zx >= zs_t ? sc * zx - lse_t : -INFINITY);",
        [(PINS, "test_log_ratio_matches_logsumexp", {}), (PINS, "test_footnote_two_token_example", {})]),
    "confidence_intercept_index": (
        "if (conf && est) conf[j] = sigmoid(est[0] * f + est[1 + j]);",
        "if (conf && est) conf[j] = sigmoid(est[0] * f + est[j]);",
        [(PINS, "test_confidence_is_sigmoid_of_affine_feature", {})]),
    # the accept rule and the draws
    "accept_test_flipped": (
        "int take = (double)u[i] < acc;", "int take = (double)u[i] > acc;",
        [(PINS, "test_footnote_two_token_example", {}), (PINS, "test_p_equals_q_accepts_everything", {})]),
    "residual_operands_transposed": (
        "r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;", "r[v] = q[v] > p[v] ? q[v] - p[v] : 0.0;",
        [(PINS, "test_footnote_two_token_example", {}), (PINS, "test_residual_inverse_cdf_brute_force", {})]),
    "cdf_boundary_inclusive": (
        "        if (c > target) {", "        if (c >= target) {",
        [(PINS, "test_uniform_at_exact_boundary_takes_next_token", {})]),
    "bonus_draw_uses_first_uniform": (
        "token = inverse_cdf(p, V, Z, (double)u[K], &mc, &fl);", "token = inverse_cdf(p, V, Z, (double)u[0], &mc, &fl);",
        [(PINS, "test_bonus_draw_follows_last_target_row", {}), (PINS, "test_cdf_output_brackets_every_draw", {})]),
    "residual_draw_uses_position_uniform": (
        "token = inverse_cdf(r, V, Z, (double)u[K], &mc, &fl);", "token = inverse_cdf(r, V, Z, (double)u[i], &mc, &fl);",
        [(PINS, "test_residual_inverse_cdf_brute_force", {}), (PINS, "test_cdf_output_brackets_every_draw", {})]),
    "greedy_emits_the_draft": (
        "if (x[i] != a) { n = i; token = a; break; }", "if (x[i] != a) { n = i; token = x[i]; break; }",
        [(PINS, "test_greedy_is_argmax_match_with_ties", {}), (TEMP, "test_low_temperature_is_greedy", {})]),
    # FLy's gate and window
    "fly_gate_tie_rejects": (
        "int open = h >= fly_theta;", "int open = h > fly_theta;",
        [(PINS, "test_fly_gate_tie_defers", {})]),
    "fly_window_one_short": (
        "for (int32_t k = j + 1; k <= j + fly_window; ++k) {", "for (int32_t k = j + 1; k < j + fly_window; ++k) {",
        [(PINS, "test_fly_truth_table_exhaustive", {"K": 3})]),
    "fly_window_fit_off_by_one": (
        "} else if (j + fly_window > Kb - 1) {", "} else if (j + fly_window > Kb - 2) {",
        [(PINS, "test_fly_truth_table_exhaustive", {"K": 3}), (PINS, "test_fly_gate_tie_defers", {})]),
    # the estimator step and the IRLS refit
    "estimator_gradient_drops_feature": (
        "            g[0] += e * f;\n", "            g[0] += e;\n",
        [(PINS, "test_estimator_hand_cases", {}), (PINS, "test_estimator_loss_and_gradient_by_finite_differences", {})]),
    "estimator_drops_rejected_label": (
        "int32_t last = n < kb ? n : kb - 1;  /* last eligible (verified) position */",
        "int32_t last = n < kb ? n - 1 : kb - 1;  /* last eligible (verified) position */",
        [(PINS, "test_estimator_hand_cases", {}), (AV, "test_pruned_labels", {})]),
    "estimator_sum_not_mean": (
        "for (int32_t k = 0; k <= K; ++k) params[k] -= lr * (g[k] / (double)N);",
        "for (int32_t k = 0; k <= K; ++k) params[k] -= lr * g[k];",
        [(PINS, "test_estimator_hand_cases", {})]),
    "estimator_label_sign": (
        "            double y = i < n ? 1.0 : 0.0;\n            double f = feature",
        "            double y = i < n ? 0.0 : 1.0;\n            double f = feature",
        [(PINS, "test_estimator_hand_cases", {})]),
    "irls_weight_dropped": (
        "double e = sg - y, w = sg * (1.0 - sg);", "double e = sg - y, w = sg;",
        [(IRLS, "test_gradient_and_hessian_by_finite_differences", {}), (IRLS, "test_hand_cases", {})]),
    "irls_damping_ignored": (
        "double step = nk > 0.0 ? d[k] * (nk / (nk + damping)) : 0.0;", "double step = nk > 0.0 ? d[k] : 0.0;",
        [(IRLS, "test_damping_scales_each_step_by_its_evidence", {"c": 7.0})]),
    "irls_step_sign": (
        "        params[k] -= step;\n", "        params[k] += step;\n",
        [(IRLS, "test_undamped_step_is_the_newton_solve", {}), (IRLS, "test_hand_cases", {})]),
    # temperature and top-p processing
    "temperature_missing_in_exponent": (
        "        p[v] = exp(sc * logit_at(row, dtype, v) - m);", "        p[v] = exp(logit_at(row, dtype, v) - m);",
        [(TEMP, "test_power_of_two_temperature_equals_scaled_logits", {"s": 2.0, "mode": oracle.STOCHASTIC}),
         (TEMP, "test_per_sequence_temperatures_apply_per_sequence", {})]),
    "nucleus_drops_boundary_ties": (
        "        if (logit_at(row, dtype, v) >= *zstar) P += p[v];", "        if (logit_at(row, dtype, v) > *zstar) P += p[v];",
        [(TOP_P, "test_ties_at_the_boundary_are_all_kept", {}), (TOP_P, "test_closed_form_four_tokens", {})]),
    # the per-position decision report and its overrides
    "imposed_decision_ignored": (
        "            if (force && force[i] >= 0) take = force[i] != 0;", "",
        [(DEC, "test_imposed_acceptance_draws_the_bonus_from_the_last_row", {}),
         (DEC, "test_imposed_rejection_draws_the_residual_of_that_row", {"i": 1})]),
    "imposed_gate_inverted": (
        "if (force && force[j] >= 0) open = force[j] != 0;", "if (force && force[j] >= 0) open = force[j] == 0;",
        [(DEC, "test_fly_imposed_gates_follow_the_window_rule", {"W": 2})]),
    "position_margin_of_the_ratio_alone": (
        "if (margin_pos) margin_pos[i] = dmin(fabs((double)u[i] - acc), mni);",
        "if (margin_pos) margin_pos[i] = dmin(acc, mni);",
        [(DEC, "test_stochastic_report_against_scipy", {})]),
    "nucleus_shift_direction_swapped": (
        "            if (shift < 0 && i > 0) *zstar = keys[i - 1].z;\n            if (shift > 0 && j < V) *zstar = keys[j].z;",
        "            if (shift > 0 && i > 0) *zstar = keys[i - 1].z;\n            if (shift < 0 && j < V) *zstar = keys[j].z;",
        [(DEC, "test_nucleus_shift_moves_the_boundary_one_group", {"shift": -1}),
         (DEC, "test_nucleus_shift_moves_the_boundary_one_group", {"shift": 1})]),
    "nucleus_doubt_bits_swapped": (
        "if (doubt) *doubt = ((mh < INFINITY || tok_hi) ? 1 : 0) | ((ml < INFINITY || tok_lo) ? 2 : 0);",
        "if (doubt) *doubt = ((mh < INFINITY || tok_hi) ? 2 : 0) | ((ml < INFINITY || tok_lo) ? 1 : 0);",
        [(DEC, "test_nucleus_doubt_bits", {})]),
    # n-gram drafting
    "ngram_shortest_first": (
        "for (int32_t n = n_max; n >= n_min && start < 0; --n) {",
        "for (int32_t n = n_min; n <= n_max && start < 0; ++n) {",
        [(NGRAM, "test_longest_match_wins_over_a_more_recent_shorter_one", {})]),
    "ngram_oldest_occurrence": (
        "for (int32_t e = L - 1; e >= n; --e) {", "for (int32_t e = n; e <= L - 1; ++e) {",
        [(NGRAM, "test_hand_cases", {})]),
    # adaptive-verification budget
    "av_ties_to_highest_index": (
        "    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);",
        "    return a->idx > b->idx ? -1 : (a->idx < b->idx ? 1 : 0);",
        [(AV, "test_cross_sequence_ties_rank_by_index", {})]),
    "av_survival_not_a_product": (
        "            sv = sv * conf[(size_t)b * K + i];", "            sv = conf[(size_t)b * K + i];",
        [(AV, "test_budget_hand_case", {})]),
}


def _compile(tmp_path, name, text):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"])
    return oracle.bind(ctypes.CDLL(str(so)))


def _run(pin):
    module, test, kwargs = pin
    getattr(importlib.import_module(module), test)(**kwargs)


def _source():
    with open(SRC) as f:
        return f.read()


def test_control_passes_every_named_pin(tmp_path, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", _compile(tmp_path, "control", _source()))
    seen = set()
    for _, _, pins in PLANTED.values():
        for pin in pins:
            key = (pin[0], pin[1], tuple(sorted(pin[2].items())))
            if key not in seen:
                seen.add(key)
                _run(pin)


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_pins_catch_the_planted_mistake(name, tmp_path, monkeypatch):
    old, new, pins = PLANTED[name]
    src = _source()
    assert src.count(old) == 1, f"the expression for {name} must occur exactly once"
    monkeypatch.setattr(oracle, "_lib", _compile(tmp_path, name, src.replace(old, new)))
    missed = []
    for pin in pins:
        try:
            _run(pin)
        except Exception:   # an assertion, or an error the mistake provokes
            continue
        missed.append(pin[1])
    assert not missed, f"{name}: these pins passed with the mistake planted: {missed}"
