"""The oracle against the values the pages print for worked examples.

Each fixture under tests/golden/ names the page and section it comes from.
"""

import math

import numpy as np
import pytest

from oracle import sampler, verify


def logits_of(probs):
    return np.log(np.asarray(probs, dtype=np.float64))


def kept_ids(keep):
    return sorted(int(i) for i in np.flatnonzero(keep))


# ---------------------------------------------------------------- sampler pins

def test_eight_word_example(golden):
    g = golden("page5_eight_words.json")
    z = np.array(g["logits"])
    p, keep, pt, _ = sampler.filtered_distribution(z, 1.0, top_p=g["top_p"])
    assert kept_ids(keep) == g["top_p_kept_ids"]
    assert abs(p[0] - g["girl_share_about"]) < g["girl_share_tolerance"]
    assert p[0] < g["top_p"] <= p[0] + p[1]
    _, keep_k, _, _ = sampler.filtered_distribution(z, 1.0, top_k=g["top_k"])
    assert kept_ids(keep_k) == g["top_k_kept_ids"]


def test_exercise_39_1(golden):
    g = golden("exercise_39_1.json")
    p = np.array(g["probs"])
    order = np.argsort(-p, kind="stable")
    assert kept_ids(sampler.keep_top_k(order, g["top_k"])) == g["top_k_kept_ids"]
    assert kept_ids(sampler.keep_top_p(order, p, g["top_p"])) == g["top_p_kept_ids"]
    # the exact-boundary case: 0.15 >= 0.30 * 0.50 holds in float64
    assert kept_ids(sampler.keep_min_p(p, g["min_p"])) == g["min_p_kept_ids"]
    # renormalisation of eq. 39.2 through the whole pipeline (logits = log p)
    _, keep, pt, _ = sampler.filtered_distribution(logits_of(p), 1.0, top_k=g["top_k"])
    np.testing.assert_allclose(pt, g["top_k_renormalised"], rtol=1e-12, atol=1e-15)
    _, keep, pt, _ = sampler.filtered_distribution(logits_of(p), 1.0, top_p=g["top_p"])
    np.testing.assert_allclose(pt, g["top_k_renormalised"], rtol=1e-12, atol=1e-15)


def test_min_p_examples(golden):
    g = golden("min_p_examples.json")
    for case in g["cases"][:2]:
        _, keep, _, _ = sampler.filtered_distribution(logits_of(case["probs"]), 1.0,
                                                      min_p=case["min_p"])
        assert kept_ids(keep) == case["kept_ids"]
    case = g["cases"][2]
    probs = np.concatenate(([0.05, 0.0051, 0.0049], np.full(200, 0.94 / 200)))
    _, keep, _, _ = sampler.filtered_distribution(logits_of(probs), 1.0, min_p=case["min_p"])
    assert all(keep[i] for i in case["kept_must_include"])
    assert not any(keep[i] for i in case["kept_must_exclude"])
    assert np.count_nonzero(keep) == 2


def test_temperature_ratio_examples(golden):
    g = golden("temperature_ratios.json")
    for case in g["cases"]:
        z = np.array([math.log(case["ratio_at_T1"]), 0.0, -1.0, -3.0])
        p, _, _, _ = sampler.filtered_distribution(z, case["T"])
        assert p[0] / p[1] == pytest.approx(case["ratio"], rel=1e-12)


# ---------------------------------------------------------------- verifier pins

def two_token(p0, q0):
    """Rows over two tokens whose token-0 probabilities are p0 and q0."""
    return logits_of([p0, 1.0 - p0]), logits_of([q0, 1.0 - q0])


def test_spec_table(golden):
    g = golden("spec_table.json")
    for row in g["rows"]:
        zp, zq = two_token(row["p"], row["q"])
        p, q = verify.softmax64(zp), verify.softmax64(zq)
        a = row["accept_prob"]
        for u in (0.0, a - 1e-9, a + 1e-9, 0.999999):
            if u < 0 or u >= 1:
                continue
            assert verify.accept_draft(p, q, 0, u) == (u < a)


def test_three_token_example(golden):
    g = golden("three_token_example.json")
    p = verify.softmax64(logits_of(g["p"]))
    q = verify.softmax64(logits_of(g["q"]))
    for x, a in enumerate(g["accept_prob"]):
        assert min(1.0, p[x] / q[x]) == pytest.approx(a, rel=1e-12)
    r = verify.residual_distribution(p, q)
    np.testing.assert_allclose(r, g["residual"], atol=g["residual_tolerance"])
    assert float(np.sum(np.minimum(p, q))) == pytest.approx(g["total_acceptance"], rel=1e-12)
    # P(output = 1): draft 1 accepted (q(1) * 1) plus rejection mass times r(1)
    reject_mass = sum(q[x] * (1.0 - min(1.0, p[x] / q[x])) for x in range(3))
    assert q[1] * 1.0 + reject_mass * r[1] == pytest.approx(g["p_out_1"], rel=1e-12)


def test_three_token_example_through_verify_row(golden):
    """The example's outcomes through the whole verify_row (K = 1)."""
    g = golden("three_token_example.json")
    zp = np.stack([logits_of(g["p"]), logits_of(g["p"])])   # position 0 and bonus
    zq = logits_of(g["q"])[None, :]
    # draft 0 with u = 0.39 is kept (accept prob 0.4); u = 0.41 rejects it
    out = verify.verify_row(zp, zq, [0], [0.39, 0.5])
    assert out["accepted"] == 1 and out["ids"][0] == 0
    out = verify.verify_row(zp, zq, [0], [0.41, 0.5])
    assert out["accepted"] == 0 and out["ids"] == [1, -1]        # 0.5 < 0.667
    out = verify.verify_row(zp, zq, [0], [0.41, 0.7])
    assert out["accepted"] == 0 and out["ids"] == [2, -1]        # 0.7 > 0.667
    # draft 1 is always kept (p/q > 1); the bonus is drawn from p with u = 0.1
    out = verify.verify_row(zp, zq, [1], [0.999, 0.1])
    assert out["accepted"] == 1 and out["ids"] == [1, 0]
