"""Plants plausible mistakes in the oracle and checks that the pins catch each.

Every mutant replaces one oracle function (on the CPU, for the duration of the
test) with a version carrying a typical slip: a wrong comparison, an off-by-one,
a swapped operand, a dropped factor.  At least one of the named pin tests must
then fail; if none does, that part of the oracle is not pinned.
"""

import numpy as np
import pytest

import oracle.beam as beam_mod
import oracle.philox as philox_mod
import oracle.prepass as prepass_mod
import oracle.sampler as sampler_mod
import oracle.verify as verify_mod
from tests import test_oracle_beam as t_beam
from tests import test_oracle_philox as t_philox
from tests import test_oracle_prepass as t_prepass
from tests import test_oracle_pins as t_pins
from tests import test_oracle_properties as t_props
from tests import test_oracle_verify_variants as t_variants
from tests.conftest import load_golden


def _softmax_times_t(z, temperature):
    x = z * float(temperature)
    w = np.exp(x - np.max(x))
    return w / np.sum(w)


def _top_k_plus_one(order, k):
    keep = np.zeros(order.size, dtype=bool)
    keep[order[: k + 1]] = True
    return keep


def _order_high_id_first(z):
    ids = np.arange(z.size)
    return np.lexsort((-ids, -z))


def _nucleus_strict(p_sorted, top_p):
    cum = np.cumsum(p_sorted)
    reached = np.flatnonzero(cum > top_p)
    return int(reached[0]) + 1 if reached.size else p_sorted.size


def _nucleus_short_by_one(p_sorted, top_p):
    cum = np.cumsum(p_sorted)
    reached = np.flatnonzero(cum >= top_p)
    return max(int(reached[0]), 1) if reached.size else p_sorted.size


def _min_p_strict(p, min_p):
    return p > float(min_p) * np.max(p)


def _min_p_absolute(p, min_p):
    return p >= float(min_p)


def _walk_ge(weights, u):
    running = np.cumsum(weights)
    past = np.flatnonzero(running >= u)
    return int(past[0]) if past.size else int(np.flatnonzero(weights > 0)[-1])


def _accept_inverted(p, q, x, u):
    return u < q[x] / max(p[x], 1e-300)


def _residual_swapped(p, q):
    r = np.maximum(q - p, 0.0)
    return r / np.sum(r) if np.sum(r) > 0 else p


def _uniform_second_word(seed, offset, row, draw):
    w1 = philox_mod.philox4x64_10((offset, row, draw, 0), (seed, 0))[1]
    return (w1 >> 11) * 2.0 ** -53


def _softmax64_times_t(row, temperature=1.0):
    z = sampler_mod.logits_to_f64(row) * float(temperature)
    w = np.exp(z - np.max(z))
    return w / np.sum(w)


def _top_token_last(row):
    z = sampler_mod.logits_to_f64(row)
    return int(np.flatnonzero(z == np.max(z))[-1])


def _top_token_of_draft_model(original):
    # greedy verification that ignores the drafts' agreement and keeps every draft
    def wrapped(p_rows, q_rows, drafts, uniforms, temperature=1.0, greedy=False, filters=None):
        if greedy or float(temperature) == 0.0:
            k = len(drafts)
            return {"accepted": k, "ids": [int(x) for x in drafts] + [verify_mod.top_token(p_rows[k])],
                    "status": 0, "accept_margin": float("inf"), "draw_margin": float("inf"),
                    "filter_margin": float("inf")}
        return original(p_rows, q_rows, drafts, uniforms, temperature, greedy, filters)
    return wrapped


def _distribution_unfiltered(row, temperature, filters):
    return verify_mod.softmax64(row, temperature), float("inf")


def _alpha_of_p_only(p_rows, q_rows, temperature=1.0, filters=None):
    return [float(np.sum(np.minimum(verify_mod.softmax64(p_rows[i], temperature), 1.0)))
            for i in range(len(q_rows))]


def _penalize_swapped(z, r, dtype="f32"):
    z, r = np.float32(z), np.float32(r)
    return np.float32(z * r) if z > 0 else np.float32(z / r)


def _allowed_inverted(words, vocab):
    ids = np.arange(vocab)
    return ((np.asarray(words, dtype=np.uint32)[ids // 32] >> (ids % 32).astype(np.uint32)) & 1) == 0


def _candidates_without_beam_score(logits, scores):
    return beam_mod.__dict__["_original_candidates"](logits, np.zeros(len(scores)))


def _log_softmax_no_norm(row):
    z = sampler_mod.logits_to_f64(row)
    return z - np.max(z)


def _fd_no_renorm(original):
    def wrapped(row, temperature, top_k=0, top_p=1.0, min_p=0.0):
        p, keep, _, diag = original(row, temperature, top_k, top_p, min_p)
        return p, keep, np.where(keep, p, 0.0), diag
    return wrapped


MUTANTS = [
    ("temperature multiplies", sampler_mod, "softmax_with_temperature", _softmax_times_t,
     [lambda: t_pins.test_temperature_ratio_examples(load_golden),
      t_props.test_temperature_ratio_identity_random]),
    ("top-k keeps k+1", sampler_mod, "keep_top_k", _top_k_plus_one,
     [lambda: t_pins.test_eight_word_example(load_golden), t_props.test_top_k_brute_force]),
    ("ties favour the higher id", sampler_mod, "descending_order", _order_high_id_first,
     [t_props.test_top_k_brute_force]),
    ("top-p uses >", sampler_mod, "nucleus_length", _nucleus_strict,
     [t_props.test_top_p_exact_boundary]),
    ("top-p one short", sampler_mod, "nucleus_length", _nucleus_short_by_one,
     [lambda: t_pins.test_eight_word_example(load_golden), t_props.test_top_p_brute_force_dyadic]),
    ("min-p uses >", sampler_mod, "keep_min_p", _min_p_strict,
     [lambda: t_pins.test_exercise_39_1(load_golden)]),
    ("min-p ignores the maximum", sampler_mod, "keep_min_p", _min_p_absolute,
     [lambda: t_pins.test_min_p_examples(load_golden)]),
    ("walk uses >=", sampler_mod, "walk", _walk_ge,
     [t_props.test_walk_boundaries]),
    ("accept ratio inverted", verify_mod, "accept_draft", _accept_inverted,
     [lambda: t_pins.test_spec_table(load_golden)]),
    ("residual max(0, q - p)", verify_mod, "residual_distribution", _residual_swapped,
     [lambda: t_pins.test_three_token_example(load_golden)]),
    ("uniform from the wrong word", philox_mod, "uniform", _uniform_second_word,
     [t_philox.test_uniform_layout]),
    ("verify temperature multiplies", verify_mod, "softmax64", _softmax64_times_t,
     [lambda: t_variants.test_temperature_acts_on_logits_over_t(0.5, 2.0),
      lambda: t_variants.test_temperature_acts_on_logits_over_t(2.0, 0.5)]),
    ("greedy ties favour the higher id", verify_mod, "top_token", _top_token_last,
     [t_variants.test_greedy_ties_go_to_the_lowest_id]),
    ("greedy keeps every draft", verify_mod, "verify_row", _top_token_of_draft_model(verify_mod.verify_row),
     [t_variants.test_greedy_emits_a_prefix_of_the_target_greedy_tokens,
      t_variants.test_greedy_ties_go_to_the_lowest_id]),
    ("verify filters dropped", verify_mod, "_distribution", _distribution_unfiltered,
     [t_variants.test_filters_with_disjoint_kept_sets_reject_every_draft,
      lambda: t_variants.test_filtered_acceptance_rate_and_output({"top_k": 2}, [4 / 7, 3 / 7, 0, 0],
                                                                   [3 / 7, 0, 4 / 7, 0])]),
    ("acceptance rate ignores q", verify_mod, "acceptance_rates", _alpha_of_p_only,
     [lambda: t_variants.test_acceptance_rate_three_token_example(load_golden),
      t_variants.test_acceptance_rate_is_one_minus_total_variation]),
    ("penalty branches swapped", prepass_mod, "penalize", _penalize_swapped,
     [t_prepass.test_penalty_branches_on_hand_values, t_prepass.test_penalty_lowers_every_score_for_r_above_one]),
    ("mask inverted", prepass_mod, "allowed_mask", _allowed_inverted,
     [t_prepass.test_masked_distribution_is_conditioned_on_the_allowed_set,
      lambda: t_prepass.test_tiny_grammar_mask("[")]),
    ("beam score ignored", beam_mod, "candidates", _candidates_without_beam_score,
     [t_beam.test_two_step_example_beats_greedy, t_beam.test_brute_force_against_log_softmax]),
    ("log-softmax without the log-sum", beam_mod, "log_softmax64", _log_softmax_no_norm,
     [t_beam.test_two_step_example_beats_greedy, t_beam.test_brute_force_against_log_softmax]),
    ("renormalisation dropped", sampler_mod, "filtered_distribution",
     _fd_no_renorm(sampler_mod.filtered_distribution),
     [lambda: t_pins.test_exercise_39_1(load_golden), t_props.test_renormalisation_invariants]),
]


beam_mod._original_candidates = beam_mod.candidates


@pytest.mark.parametrize("name,module,attr,mutant,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, module, attr, mutant, pins):
    monkeypatch.setattr(module, attr, mutant)
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught += 1
    assert caught == len(pins), f"mutant '{name}' slipped past {len(pins) - caught} pin(s)"


def test_wrong_philox_multiplier_is_caught(monkeypatch):
    monkeypatch.setattr(philox_mod, "PHILOX_M0", philox_mod.PHILOX_M0 ^ 2)
    with pytest.raises(AssertionError):
        t_philox.test_random_blocks_match_numpy()
