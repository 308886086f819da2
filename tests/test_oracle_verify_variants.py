"""Pins of the verifier oracle's variants: temperature on p and q, and greedy
verification ("Speculative decoding -- Hinglish notes", section "Temperature
and Sampling"; "Inference: Sampling, the KV Cache, Speculative Decoding and
int8", section "Speculative decoding").

Each pin rests on something the pages or the mathematics fix, not on the
oracle's own formulas:
* greedy verification emits a prefix of the target's own greedy tokens (the
  pages: its output is identical to plain greedy decoding with the target);
* greedy verification is the T -> 0 limit of the stochastic rule when the
  drafts are the draft model's greedy tokens (one-hot p and q);
* softmax(z / T) depends on z / T only: T = 1/2 on z equals T = 1 on 2 z, and
  T = 2 on z equals T = 1 on z / 2, exactly (powers of two);
* with p = q every draft is kept at any temperature (ratio exactly 1).
"""

import numpy as np
import pytest

from oracle import philox
from oracle import verify as over


def batch(b, k, v, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    p = (rng.standard_normal((b, k + 1, v)) * scale).astype(np.float32)
    q = (rng.standard_normal((b, k, v)) * scale).astype(np.float32)
    return p, q


def targets_greedy(p_rows):
    return [over.top_token(r) for r in p_rows]


def test_greedy_emits_a_prefix_of_the_target_greedy_tokens():
    b, k, v = 40, 5, 64
    p, q = batch(b, k, v, seed=1)
    rng = np.random.default_rng(2)
    drafts = rng.integers(0, v, (b, k))
    # make the first m drafts of row r the target's greedy tokens, m = r % (k + 1)
    for r in range(b):
        tops = targets_greedy(p[r])
        m = r % (k + 1)
        drafts[r, :m] = tops[:m]
        if m < k and drafts[r, m] == tops[m]:
            drafts[r, m] = (tops[m] + 1) % v
    res = over.spec_verify(p, q, drafts, seed=0, offset=0, greedy=True)
    for r, out in enumerate(res):
        tops = targets_greedy(p[r])
        m = r % (k + 1)
        assert out["accepted"] == m
        emitted = out["ids"][: m + 1]
        assert emitted == tops[: m + 1]          # the target's greedy tokens
        assert out["ids"][m + 1:] == [-1] * (k - m)
    # temperature 0 is the same rule
    res0 = over.spec_verify(p, q, drafts, seed=0, offset=0, temperature=0.0)
    assert [x["ids"] for x in res0] == [x["ids"] for x in res]


def test_greedy_is_the_zero_temperature_limit():
    b, k, v = 30, 4, 48
    p, q = batch(b, k, v, seed=3)
    # separate every row's maximum by at least 1, so that T = 2^-10 gives exact one-hots
    for arr in (p, q):
        for idx in np.ndindex(arr.shape[:2]):
            row = arr[idx]
            row[np.argmax(row)] = np.max(row) + 1.0
    drafts = np.array([[over.top_token(q[r, i]) for i in range(k)] for r in range(b)])
    # some drafts agree with the target by construction
    for r in range(0, b, 3):
        for i in range(k):
            q[r, i] = p[r, i][: v]
        drafts[r] = [over.top_token(p[r, i]) for i in range(k)]
    cold = over.spec_verify(p, q, drafts, seed=5, offset=2, temperature=2.0 ** -10)
    greedy = over.spec_verify(p, q, drafts, seed=5, offset=2, greedy=True)
    assert [x["ids"] for x in cold] == [x["ids"] for x in greedy]
    assert [x["accepted"] for x in cold] == [x["accepted"] for x in greedy]
    assert any(x["accepted"] == k for x in greedy) and any(x["accepted"] < k for x in greedy)


@pytest.mark.parametrize("t, factor", [(0.5, 2.0), (2.0, 0.5)])
def test_temperature_acts_on_logits_over_t(t, factor):
    b, k, v = 24, 4, 40
    p, q = batch(b, k, v, seed=7, scale=1.5)
    drafts = np.random.default_rng(8).integers(0, v, (b, k))
    hot = over.spec_verify(p, q, drafts, seed=1, offset=3, temperature=t)
    scaled = over.spec_verify((p * np.float32(factor)).astype(np.float32),
                              (q * np.float32(factor)).astype(np.float32), drafts, seed=1, offset=3)
    assert [x["ids"] for x in hot] == [x["ids"] for x in scaled]
    assert [x["accepted"] for x in hot] == [x["accepted"] for x in scaled]
    # and the temperature matters: T = 1 on z gives other results somewhere
    cool = over.spec_verify(p, q, drafts, seed=1, offset=3)
    assert [x["ids"] for x in cool] != [x["ids"] for x in hot]


@pytest.mark.parametrize("t", [0.3, 1.0, 2.5])
def test_equal_distributions_keep_every_draft(t):
    b, k, v = 16, 5, 32
    p, _ = batch(b, k, v, seed=11)
    q = p[:, :k].copy()
    drafts = np.random.default_rng(12).integers(0, v, (b, k))
    res = over.spec_verify(p, q, drafts, seed=2, offset=0, temperature=t)
    for r, out in enumerate(res):
        assert out["accepted"] == k
        assert out["ids"][:k] == [int(x) for x in drafts[r]]
        # the bonus is the walk of p_K at temperature t with draw K
        u = philox.uniform(2, 0, r, k)
        assert out["ids"][k] == over.walk(over.softmax64(p[r, k], t), u)


def test_greedy_ties_go_to_the_lowest_id():
    # np.argmax returns the first occurrence of the maximum: the textbook
    # arg-max with the lowest id on ties, which greedy decoding follows
    b, k, v = 12, 3, 20
    rng = np.random.default_rng(13)
    p = rng.integers(-3, 3, (b, k + 1, v)).astype(np.float32)   # many ties
    q = rng.integers(-3, 3, (b, k, v)).astype(np.float32)
    for r in range(b):
        for i in range(k + 1):
            assert over.top_token(p[r, i]) == int(np.argmax(p[r, i]))
    drafts = np.array([[int(np.argmax(p[r, i])) for i in range(k)] for r in range(b)])
    drafts[::2, 1] = (drafts[::2, 1] + 1) % v        # a mismatch at position 1 in even rows
    res = over.spec_verify(p, q, drafts, seed=0, offset=0, greedy=True)
    for r, out in enumerate(res):
        want = [int(np.argmax(p[r, i])) for i in range(k + 1)]
        if r % 2 == 0:
            assert out["accepted"] == 1 and out["ids"] == want[:2] + [-1] * (k - 1)
        else:
            assert out["accepted"] == k and out["ids"] == want


def test_per_row_knobs():
    # row_mode follows the sampler's knob rules; the verifier applies no filter
    from spec_verify_gb300 import workloads
    b, k, v = 10, 2, 30
    p, q = batch(b, k, v, seed=17)
    q[3] = np.nan                      # greedy rows never look at q
    drafts = np.random.default_rng(18).integers(0, v, (b, k))
    prm = workloads.make_params(b)
    prm["temperature"][1] = 0.5
    prm["greedy"][2] = 1
    prm["temperature"][3] = 0.0
    prm["temperature"][4] = -0.5
    prm["top_k"][5] = 3
    prm["top_p"][6] = 0.5
    prm["min_p"][7] = 0.2
    prm["top_k"][8] = v                # top_k >= V is off
    prm["temperature"][9] = np.nan
    res = over.spec_verify(p, q, drafts, 3, 1, params=prm)
    status = [r["status"] for r in res]
    assert status == [0, 0, 0, 0, 1, 0, 0, 0, 0, 1]   # rows 5..7 filtered, row 8 off
    assert all(r["accepted"] == -1 and r["ids"] == [-1] * (k + 1) for r in res if r["status"])
    same = over.spec_verify(p, q, drafts, 3, 1, rows=[0, 8])
    assert [r["ids"] for r in same] == [res[0]["ids"], res[8]["ids"]]
    assert res[1]["ids"] == over.spec_verify(p, q, drafts, 3, 1, rows=[1], temperature=0.5)[0]["ids"]
    for r in (2, 3):
        assert res[r]["ids"] == over.spec_verify(p, q, drafts, 3, 1, rows=[r], greedy=True)[0]["ids"]
    assert over.row_mode(prm[5], v)[3] == (3, 1.0, 0.0)
    assert over.row_mode(prm[8], v)[3] is None


# ------------------------------------------------------------------ filters on p and q
#
# Hand-computed kept sets on four tokens with p = (.4, .3, .2, .1):
#   top_k = 2   keeps {0, 1}:    p~ = (4/7, 3/7, 0, 0)
#   min_p = 0.45 keeps p >= .18: p~ = (4/9, 3/9, 2/9, 0)
#   top_p = 0.75 keeps .4+.3+.2: p~ = (4/9, 3/9, 2/9, 0)

P4 = np.log([0.4, 0.3, 0.2, 0.1])
CHI2_999 = {1: 10.83, 2: 13.82, 3: 16.27}


def _tiled(rows, *dists):
    return np.tile(np.stack(dists).astype(np.float32), (rows, 1, 1))


def _drafts_from_filtered_q(Q, prm_one, seed=1):
    from oracle import sampler as osam
    b, k, v = Q.shape
    prm = np.repeat(prm_one, b * k)
    res = osam.sample(Q.reshape(b * k, v), prm, seed, 0)
    return np.array([r["token"] for r in res], dtype=np.int32).reshape(b, k)


def _chi2(counts, probs):
    probs = np.asarray(probs, dtype=np.float64)
    mask = probs > 0
    assert np.all(counts[~mask] == 0)
    exp = probs[mask] * counts.sum()
    return float(np.sum((counts[mask] - exp) ** 2 / exp)), int(mask.sum()) - 1


def test_filters_with_disjoint_kept_sets_reject_every_draft():
    # q = (.1, .2, .3, .4) with top_k = 2 keeps {2, 3}, p keeps {0, 1}: sum min(p~, q~) = 0,
    # so no draft is kept and the replacement follows p~ = (4/7, 3/7, 0, 0).  Filtering
    # only one side would keep some drafts (sum min = 0.3 either way).
    from spec_verify_gb300 import workloads
    rows = 6000
    prm = workloads.make_params(1, top_k=2)
    P = _tiled(rows, P4, P4)
    Q = _tiled(rows, np.log([0.1, 0.2, 0.3, 0.4]))
    drafts = _drafts_from_filtered_q(Q, prm)
    assert set(np.unique(drafts)) <= {2, 3}
    res = over.spec_verify(P, Q, drafts, 4, 0, params=np.repeat(prm, rows))
    assert all(r["accepted"] == 0 for r in res)
    counts = np.bincount([r["ids"][0] for r in res], minlength=4)
    stat, dof = _chi2(counts, [4 / 7, 3 / 7, 0, 0])
    assert stat < CHI2_999[dof]


@pytest.mark.parametrize("knob, p_tilde, q_tilde", [
    ({"top_k": 2}, [4 / 7, 3 / 7, 0, 0], [3 / 7, 0, 4 / 7, 0]),
    ({"min_p": 0.45}, [4 / 9, 3 / 9, 2 / 9, 0], [3 / 9, 0, 4 / 9, 2 / 9]),
    ({"top_p": 0.75}, [4 / 9, 3 / 9, 2 / 9, 0], [3 / 9, 0, 4 / 9, 2 / 9]),
])
def test_filtered_acceptance_rate_and_output(knob, p_tilde, q_tilde):
    # q = (.3, .1, .4, .2): with K = 1 the mean accepted length is
    # alpha = sum min(p~, q~) ("Decoding & Speculative Sampling", section 39.4),
    # and both emitted positions follow p~ (the bonus row is p again).
    from spec_verify_gb300 import workloads
    rows = 12000
    prm = workloads.make_params(1, **knob)
    P = _tiled(rows, P4, P4)
    Q = _tiled(rows, np.log([0.3, 0.1, 0.4, 0.2]))
    drafts = _drafts_from_filtered_q(Q, prm)
    res = over.spec_verify(P, Q, drafts, 5, 0, params=np.repeat(prm, rows))
    acc = np.array([r["accepted"] for r in res])
    ids = np.array([r["ids"] for r in res])
    alpha = float(np.sum(np.minimum(p_tilde, q_tilde)))
    assert abs(acc.mean() - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / rows)
    for pos in (0, 1):
        reached = acc >= pos
        stat, dof = _chi2(np.bincount(ids[reached, pos], minlength=4), p_tilde)
        assert stat < CHI2_999[dof], (pos, stat)


def test_top_k_one_is_greedy_verification():
    # top_k = 1 leaves one-hot p~ and q~ at the arg-max: a draft is kept iff it
    # is the target's top token, and the replacement or bonus is that token.
    from spec_verify_gb300 import workloads
    b, k, v = 30, 4, 25
    p, q = batch(b, k, v, seed=19)
    rng = np.random.default_rng(20)
    drafts = rng.integers(0, v, (b, k))
    for r in range(0, b, 2):
        m = r % (k + 1)
        drafts[r, :m] = [over.top_token(p[r, i]) for i in range(m)]
    top1 = over.spec_verify(p, q, drafts, 6, 0, params=workloads.make_params(b, top_k=1, temperature=0.7))
    greedy = over.spec_verify(p, q, drafts, 6, 0, greedy=True)
    assert [x["ids"] for x in top1] == [x["ids"] for x in greedy]
    assert any(x["accepted"] > 0 for x in greedy)


# ------------------------------------------------------------------ acceptance rates


def test_acceptance_rate_three_token_example(golden):
    # the page's example: p = (.2, .5, .3), q = (.5, .3, .2), total acceptance 0.7
    g = golden("three_token_example.json")
    p = np.log(np.array(g["p"]))[None].astype(np.float64)
    q = np.log(np.array(g["q"]))[None].astype(np.float64)
    assert abs(over.acceptance_rates(np.concatenate([p, p]), q)[0] - g["total_acceptance"]) < 1e-12


def test_acceptance_rate_is_one_minus_total_variation():
    # sum min(p, q) = 1 - (1/2) sum |p - q| for any two distributions
    b, k, v = 6, 3, 50
    p, q = batch(b, k, v, seed=23)
    for r in range(b):
        for t in (0.6, 1.0, 1.7):
            got = over.acceptance_rates(p[r], q[r], t)
            for i in range(k):
                pi, qi = over.softmax64(p[r, i], t), over.softmax64(q[r, i], t)
                assert abs(got[i] - (1.0 - 0.5 * np.sum(np.abs(pi - qi)))) < 1e-12


def test_acceptance_rate_matches_simulated_acceptance():
    # with K = 1 and drafts drawn from q, the accepted fraction estimates alpha_0
    rows, v = 20000, 6
    rng = np.random.default_rng(29)
    zp = rng.normal(0, 1.2, (2, v)).astype(np.float32)
    zq = rng.normal(0, 1.2, (1, v)).astype(np.float32)
    P = np.tile(zp, (rows, 1, 1))
    Q = np.tile(zq, (rows, 1, 1))
    drafts = _drafts_from_filtered_q(Q, _unit_params())
    res = over.spec_verify(P, Q, drafts, 8, 0, rows=range(rows), alpha=True)
    alpha = res[0]["alpha"][0]
    assert all(r["alpha"] == [alpha] for r in res[:5])
    acc = np.mean([r["accepted"] for r in res])
    assert abs(acc - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / rows)


def _unit_params():
    from spec_verify_gb300 import workloads
    return workloads.make_params(1)


def test_acceptance_rate_filtered_and_undefined_rows():
    from spec_verify_gb300 import workloads
    rows = 3
    P = _tiled(rows, P4, P4)
    Q = _tiled(rows, np.log([0.3, 0.1, 0.4, 0.2]))
    prm = workloads.make_params(rows, top_k=2)
    prm["greedy"][1] = 1
    prm["temperature"][2] = -1.0
    res = over.spec_verify(P, Q, np.zeros((rows, 1), dtype=np.int32), 0, 0, params=prm, alpha=True)
    assert abs(res[0]["alpha"][0] - 3 / 7) < 1e-7      # float32 logits; sum min((4/7, 3/7, 0, 0), (3/7, 0, 4/7, 0))
    assert np.isnan(res[1]["alpha"][0]) and np.isnan(res[2]["alpha"][0])


def test_exercise_39_2_residual_mass_is_one_minus_acceptance():
    # "Decoding & Speculative Sampling", Exercise 39.2: for normalised p and q,
    # sum_x max(0, p(x) - q(x)) = 1 - sum_x min(p(x), q(x)); the rejection path
    # therefore carries exactly the residual mass
    b, k, v = 5, 3, 40
    p, q = batch(b, k, v, seed=31)
    for r in range(b):
        alphas = over.acceptance_rates(p[r], q[r], 0.8)
        for i in range(k):
            pi, qi = over.softmax64(p[r, i], 0.8), over.softmax64(q[r, i], 0.8)
            assert abs(np.sum(np.maximum(0.0, pi - qi)) - (1.0 - alphas[i])) < 1e-12
