"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source to a temporary directory, plants one
plausible mistake (a dropped term, a wrong sign, a wrong index, a transposed
operand, a wrong tie-break), compiles it with gcc and runs the pin that should
catch it against the mutant.  The pins are only worth trusting if every mutant
fails at least one of them.  Nothing here touches a GPU.
"""

import os
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dspark_oracle.c")

MUTANTS = [
    # (name, original text, planted text, pins expected to catch it)
    ("predecessor-not-carried", "      prev = best;\n", "      prev = anchors[b];\n",
     ["test_sampler_matches_exhaustive_joint", "test_greedy_is_argmax_of_calibrated_logits"]),
    ("block-race-exponential-not-logged", "const double score = log(Z) - log(E);",
     "const double score = log(Z) - E;", ["test_temperature_scales_the_sampled_softmax"]),
    ("stage2-reuses-stage1-uniform", "race_u2(seed, b, k, bblk, tag0) * bestZ",
     "race_u1(seed, b, k, bblk, tag0) * bestZ",
     ["test_temperature_scales_the_sampled_softmax"]),
    ("block-mass-drops-first-token",
     "while (j < n && ((uint32_t)(ids ? ids[j] : j) >> 4) == blk) Z += w[j++];",
     "while (j < n && ((uint32_t)(ids ? ids[j] : j) >> 4) == blk) { if (j > i) Z += w[j]; ++j; }",
     ["test_temperature_scales_the_sampled_softmax", "test_sampler_matches_exhaustive_joint"]),
    ("w2-transposed", "l[v] += ei * bf16_to_double(w2row[v]);",
     "l[v] += ei * bf16_to_double(W2[(int64_t)v * r + i]);",
     ["test_teacher_forced_logits_match_numpy"]),
    ("philox-9-rounds", "round < 10; ++round", "round < 9; ++round",
     ["test_philox_known_answers"]),
    ("logprob-without-temperature", "logprobs[o] = l[best] / Tp - lse;",
     "logprobs[o] = l[best] - lse;", ["test_temperature_scales_the_sampled_softmax"]),
    ("bias-dropped", "l[v] = (double)Urow[v] + l[v];", "l[v] = (double)Urow[v];",
     ["test_teacher_forced_logits_match_numpy", "test_np_torch_worked_example"]),
    ("topk-ties-to-larger-id", "while (p > 0 && x > vals[p - 1])",
     "while (p > 0 && x >= vals[p - 1])", ["test_topk_matches_lexsort"]),
    ("pair-predecessor-same-position", "cand[(bt - 1) * topk + i]", "cand[bt * topk + i]",
     ["test_pair_scores_match_numpy", "test_walk_with_k_equal_V_is_the_full_head"]),
    ("confidence-uses-current-token", "tokens[(int64_t)b * K + k - 1]", "tokens[(int64_t)b * K + k]",
     ["test_confidence_closed_form"]),
    ("gate-without-sigmoid", "for (int i = 0; i < r; ++i) acc[i] = sigmoid(acc[i]);", "",
     ["test_gate_matches_numpy"]),
    ("walk-slot-not-carried", "      slot = next;\n", "      slot = 0;\n",
     ["test_walk_with_k_equal_V_is_the_full_head"]),
    ("uniform-offset", "+ 0.5) * (1.0 / 8388608.0)", "+ 1.0) * (1.0 / 8388608.0)",
     ["test_uniform_grid_and_word_selection"]),
    ("schedule-batch-size-off-by-one", "const double next = (sum + c[i].a) * sps[R + i + 1];",
     "const double next = (sum + c[i].a) * sps[R + i];",
     ["test_schedule_stops_at_the_first_dip_of_a_jagged_curve",
      "test_schedule_matches_exhaustive_search_when_theta_is_unimodal"]),
    ("schedule-ranks-ascending", "if (x->a != y->a) return x->a > y->a;",
     "if (x->a != y->a) return x->a < y->a;",
     ["test_schedule_matches_exhaustive_search_when_theta_is_unimodal"]),
    ("verify-ratio-inverted", "fmin(1.0, pv[x] / qv[x])", "fmin(1.0, qv[x] / pv[x])",
     ["test_verify_commits_the_target_distribution"]),
    ("verify-resample-from-target", "z[v] = d > 0.0 ? log(d) : -INFINITY;",
     "z[v] = pv[v] > 0.0 ? log(pv[v]) : -INFINITY;",
     ["test_verify_commits_the_target_distribution",
      "test_verify_greedy_draft_accepts_with_the_target_probability"]),
    ("verify-bonus-row-before-the-window", "target_probs(P + ((int64_t)b * (K + 1) + L) * V, V, Tt, pv);",
     "target_probs(P + ((int64_t)b * (K + 1) + (L > 0 ? L - 1 : 0)) * V, V, Tt, pv);",
     ["test_verify_target_equal_to_draft_accepts_every_token"]),
    ("label-overlap-by-max", "s += fmin(pv[v], qv[v]);", "s += fmax(pv[v], qv[v]);",
     ["test_accept_label_special_cases", "test_accept_label_is_the_verifier_acceptance_rate"]),
    ("sts-targets-not-cumulative", "y[n] *= (double)label[(int64_t)n * K + k];",
     "y[n] = (double)label[(int64_t)n * K + k];",
     ["test_sts_recovers_the_generating_temperatures", "test_sts_matches_a_dense_scan"]),
    ("sts-survival-not-carried", "for (int n = 0; n < N; ++n) a[n] *= sigmoid(z[n] / tau[k]);", "",
     ["test_sts_recovers_the_generating_temperatures", "test_sts_matches_a_dense_scan"]),
    ("sts-temperature-inverted", "const double L = sts_loss(z, a, y, N, exp(-x));",
     "const double L = sts_loss(z, a, y, N, exp(x));",
     ["test_sts_recovers_the_generating_temperatures"]),
    ("confidence-temperature-ignored", "sigmoid(tau ? z / tau[k] : z)", "sigmoid(z)",
     ["test_confidence_applies_per_position_temperatures"]),
    ("label-predecessor-not-carried", "      label[(int64_t)b * K + k] = s;\n      prev = x;\n",
     "      label[(int64_t)b * K + k] = s;\n",
     ["test_accept_label_special_cases", "test_accept_label_is_the_verifier_acceptance_rate"]),
    ("rnn-state-not-carried", "s[i] = Arow[i] * s[i] + (Grow ? w1 * Grow[i] : w1);",
     "s[i] = (Grow ? w1 * Grow[i] : w1);",
     ["test_rnn_state_is_a_geometric_series_under_constant_decay",
      "test_rnn_unrolled_state_matches_teacher_forced_logits"]),
    ("rnn-decay-on-the-input", "s[i] = Arow[i] * s[i] + (Grow ? w1 * Grow[i] : w1);",
     "s[i] = s[i] + Arow[i] * (Grow ? w1 * Grow[i] : w1);",
     ["test_rnn_state_is_a_geometric_series_under_constant_decay",
      "test_rnn_with_zero_decay_is_the_markov_head"]),
    ("rnn-input-gate-ignored", "s[i] = Arow[i] * s[i] + (Grow ? w1 * Grow[i] : w1);",
     "s[i] = Arow[i] * s[i] + w1;",
     ["test_rnn_unrolled_state_matches_teacher_forced_logits",
      "test_rnn_with_zero_decay_is_the_markov_head"]),
    ("rnn-state-not-reset-per-request", "    for (int i = 0; i < r; ++i) e[i] = 0.0; /* s_{-1} = 0 */",
     "", ["test_rnn_sampler_matches_exhaustive_joint"]),
    ("rnn-draft-predecessor-not-carried", "      prev = best;\n", "      prev = anchors[b];\n",
     ["test_rnn_sampler_matches_exhaustive_joint"]),
]


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in the oracle source"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", str(so), str(c), "-lm"], check=True)
    return oracle.Oracle(str(so))


def _run_pin(fn_name, orc):
    fn = getattr(pins, fn_name)
    marks = getattr(fn, "pytestmark", [])
    params = [m for m in marks if m.name == "parametrize"]
    combos = [{}]
    for m in params:
        names = [n.strip() for n in m.args[0].split(",")]
        new = []
        for c in combos:
            for val in m.args[1]:
                vals = val if len(names) > 1 else (val,)
                new.append({**c, **dict(zip(names, vals))})
        combos = new
    for kw in combos:
        fn(orc, **kw)


@pytest.mark.parametrize("name,old,new,catchers", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, catchers):
    mutant = _compile(tmp_path, name, old, new)
    caught = []
    for pin in catchers:
        try:
            _run_pin(pin, mutant)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin)
    assert caught, f"planted mistake '{name}' passed every pin in {catchers}"


def test_unmutated_source_passes_the_same_pins(tmp_path):
    clean = _compile(tmp_path, "clean", "dspark_oracle", "dspark_oracle")
    for *_, catchers in MUTANTS:
        for pin in catchers:
            _run_pin(pin, clean)
