"""The oracle against closed forms, invariants and brute force.

Nothing here retypes the oracle's formulas: each check is an independent
characterisation (subset enumeration, exactness of speculative sampling,
closed-form expectations, chi-square against the target distribution).
"""

import itertools
import math

import numpy as np
import pytest

from oracle import philox, sampler, verify
from spec_verify_gb300 import workloads


def lex_greater(z, i, j):
    """(z_i, -i) > (z_j, -j): token i precedes token j in the kept order."""
    return z[i] > z[j] or (z[i] == z[j] and i < j)


# ------------------------------------------------------------------ top-k

def test_top_k_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(300):
        vocab = int(rng.integers(2, 13))
        z = np.round(rng.normal(0, 1.5, size=vocab), 1)      # many exact ties
        k = int(rng.integers(1, vocab))
        _, keep, _, _ = sampler.filtered_distribution(z, 1.0, top_k=k)
        assert np.count_nonzero(keep) == k
        for i in np.flatnonzero(keep):
            for j in np.flatnonzero(~keep):
                assert lex_greater(z, i, j)


# ------------------------------------------------------------------ top-p

def test_top_p_brute_force_dyadic():
    """Shortest subset reaching top_p, on dyadic probabilities (exact sums)."""
    rng = np.random.default_rng(2)
    for _ in range(200):
        vocab = int(rng.integers(2, 10))
        counts = rng.multinomial(64, rng.dirichlet(np.ones(vocab)))
        if np.count_nonzero(counts) == 0:
            continue
        p = counts / 64.0
        top_p = int(rng.integers(1, 64)) / 64.0
        order = np.lexsort((np.arange(vocab), -p))
        keep = sampler.keep_top_p(order, p, top_p)
        size = np.count_nonzero(keep)
        reach = [m for m in range(1, vocab + 1)
                 if any(sum(p[list(s)]) >= top_p for s in itertools.combinations(range(vocab), m))]
        assert size == reach[0]
        # the kept tokens are the most likely ones
        assert np.min(p[keep]) >= np.max(p[~keep], initial=-1.0)


def test_top_p_exact_boundary():
    """Cumulative sum exactly equal to top_p stops there (">=", shortest prefix)."""
    p = np.array([0.5, 0.25, 0.25])
    order = np.arange(3)
    assert sampler.nucleus_length(p[order], 0.75) == 2
    assert sampler.nucleus_length(p[order], 0.75 + 1e-12) == 3
    assert sampler.nucleus_length(p[order], 0.5) == 1
    assert sampler.nucleus_length(p[order], 0.0) == 1          # never empty


def test_filters_intersect_as_shortest_prefix():
    rng = np.random.default_rng(3)
    for _ in range(200):
        vocab = int(rng.integers(3, 40))
        z = np.round(rng.normal(0, 2, size=vocab), 1)
        t, k = float(rng.uniform(0.3, 2.0)), int(rng.integers(0, vocab + 1))
        tp, mp = float(rng.choice([1.0, 0.5, 0.9])), float(rng.choice([0.0, 0.05, 0.3]))
        _, keep, _, _ = sampler.filtered_distribution(z, t, k, tp, mp)
        sizes = []
        for kw in ({"top_k": k}, {"top_p": tp}, {"min_p": mp}):
            _, single, _, _ = sampler.filtered_distribution(z, t, **kw)
            sizes.append(np.count_nonzero(single))
            assert np.all(single[keep])            # S is inside every mask
        assert np.count_nonzero(keep) == min(sizes)
        order = sampler.descending_order(z)
        assert np.all(keep[order[: np.count_nonzero(keep)]])   # a prefix


# ------------------------------------------------------------------ temperature, eq. 39.2

def test_temperature_ratio_identity_random():
    rng = np.random.default_rng(4)
    for _ in range(50):
        z = rng.normal(0, 2, size=20)
        p1, _, _, _ = sampler.filtered_distribution(z, 1.0)
        t = float(rng.uniform(0.3, 3.0))
        pt, _, _, _ = sampler.filtered_distribution(z, t)
        i, j = rng.choice(20, size=2, replace=False)
        assert pt[i] / pt[j] == pytest.approx((p1[i] / p1[j]) ** (1.0 / t), rel=1e-9)


def test_renormalisation_invariants():
    rng = np.random.default_rng(5)
    for _ in range(100):
        z = rng.normal(0, 2, size=50)
        p, keep, pt, _ = sampler.filtered_distribution(z, 0.8, top_k=10, top_p=0.9, min_p=0.02)
        assert math.isclose(float(np.sum(pt)), 1.0, rel_tol=1e-12)
        assert np.all(pt[~keep] == 0.0)
        kept = np.flatnonzero(keep)
        ratio = pt[kept] / p[kept]
        assert np.allclose(ratio, ratio[0], rtol=1e-12)      # p~ proportional to p on S


# ------------------------------------------------------------------ greedy and the draw

def test_greedy_is_low_temperature_limit():
    rng = np.random.default_rng(6)
    for _ in range(50):
        z = rng.normal(0, 3, size=64)
        top = np.argsort(-z)
        if z[top[0]] - z[top[1]] < 1.0:
            z[top[0]] = z[top[1]] + 1.0
        argmax = int(np.argmax(z))
        for u in (1e-9, 0.5, 0.999999999):
            assert sampler.sample_row(z, 0.01, 0, 1.0, 0.0, 0, u)["token"] == argmax
        greedy = sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 1, 0.7)
        assert greedy["token"] == argmax and greedy["prob"] == 1.0
        assert sampler.sample_row(z, 0.0, 0, 1.0, 0.0, 0, 0.7)["token"] == argmax


def test_greedy_ties_take_lowest_id():
    z = np.array([1.0, 3.0, -2.0, 3.0, 3.0])
    assert sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 1, 0.3)["token"] == 1


def test_walk_boundaries():
    assert sampler.walk(np.array([0.25, 0.25, 0.5]), 0.25) == 1       # strictly passes u
    assert sampler.walk(np.array([0.25, 0.25, 0.5]), 0.0) == 0
    assert sampler.walk(np.array([0.0, 0.5, 0.0, 0.5]), 0.0) == 1     # zero mass never drawn
    assert sampler.walk(np.array([0.0, 0.5, 0.0, 0.5]), 0.5) == 3
    assert sampler.walk(np.array([0.5, 0.5, 0.0]), 1.0) == 1          # past the end: last kept


def chi2_stat(counts, probs):
    expected = probs * counts.sum()
    mask = expected > 0
    assert np.all(counts[~mask] == 0)
    return float(np.sum((counts[mask] - expected[mask]) ** 2 / expected[mask])), int(mask.sum()) - 1


CHI2_999 = {1: 10.83, 2: 13.82, 3: 16.27, 4: 18.47, 5: 20.52, 6: 22.46, 7: 24.32}


def test_draw_follows_renormalised_distribution():
    z = np.array([2.0, 1.0, 0.5, 0.0, -1.0, -3.0])
    rows = 20000
    logits = np.tile(z.astype(np.float32), (rows, 1))
    params = workloads.make_params(rows, temperature=0.9, top_k=5, top_p=0.97)
    results = sampler.sample(logits, params, seed=3, offset=1)
    _, _, pt, _ = sampler.filtered_distribution(z, 0.9, top_k=5, top_p=0.97)
    counts = np.bincount([r["token"] for r in results], minlength=z.size)
    stat, dof = chi2_stat(counts, pt)
    assert stat < CHI2_999[dof]


# ------------------------------------------------------------------ verifier

def exactness_by_quadrature(p_probs, q_probs, n=4000):
    """P(output = y) of one verify position, integrated over u on midpoint grids.

    Accept fractions come from verify_row with each draft x, the replacement
    distribution from verify_row forced to reject (u just below 1).
    """
    zp = np.log(np.asarray(p_probs))
    zq = np.log(np.asarray(q_probs))
    vocab = zp.size
    p_rows = np.stack([zp, zp])
    q_rows = zq[None, :]
    grid = (np.arange(n) + 0.5) / n
    p = verify.softmax64(zp)
    q = verify.softmax64(zq)
    accept = np.zeros(vocab)
    for x in range(vocab):
        accept[x] = np.mean([verify.verify_row(p_rows, q_rows, [x], [u, 0.5])["accepted"] == 1
                             for u in grid])
    rejecting = [x for x in range(vocab) if p[x] < q[x]]
    replace = np.zeros(vocab)
    if rejecting:
        x = rejecting[0]
        for u2 in grid:
            out = verify.verify_row(p_rows, q_rows, [x], [1.0 - 1e-12, u2])
            assert out["accepted"] == 0
            replace[out["ids"][0]] += 1.0 / n
    return sum(q[x] * (accept[x] * np.eye(vocab)[x] + (1 - accept[x]) * replace)
               for x in range(vocab))


def test_verify_exactness_three_token_example(golden):
    g = golden("three_token_example.json")
    out = exactness_by_quadrature(g["p"], g["q"])
    np.testing.assert_allclose(out, g["p"], atol=2e-3)


def test_verify_exactness_random_pairs():
    rng = np.random.default_rng(8)
    for _ in range(3):
        p = rng.dirichlet(np.ones(5))
        q = rng.dirichlet(np.ones(5) * 0.5)
        out = exactness_by_quadrature(p, q, n=3000)
        np.testing.assert_allclose(out, p, atol=3e-3)


def draft_from_oracle(q_logits, seed, offset):
    """Draft ids drawn from q (T = 1, no filters) with the oracle sampler."""
    b, k, v = q_logits.shape
    flat = q_logits.reshape(b * k, v)
    params = workloads.make_params(b * k)
    res = sampler.sample(flat, params, seed=seed, offset=offset)
    return np.array([r["token"] for r in res], dtype=np.int32).reshape(b, k)


@pytest.mark.slow
def test_verify_chi_square_v8():
    """Every emitted token follows the target distribution of its position."""
    rng = np.random.default_rng(9)
    vocab, k, rows = 8, 2, 12000
    zp = rng.normal(0, 1.5, size=(k + 1, vocab)).astype(np.float32)
    zq = rng.normal(0, 1.5, size=(k, vocab)).astype(np.float32)       # a different draft
    P = np.tile(zp, (rows, 1, 1))
    Q = np.tile(zq, (rows, 1, 1))
    drafts = draft_from_oracle(Q, seed=1, offset=0)
    res = verify.spec_verify(P, Q, drafts, seed=0, offset=0)
    ids = np.array([r["ids"] for r in res])
    acc = np.array([r["accepted"] for r in res])
    for pos in range(k + 1):
        reached = acc >= pos
        counts = np.bincount(ids[reached, pos], minlength=vocab)
        stat, dof = chi2_stat(counts, verify.softmax64(zp[pos]))
        assert stat < CHI2_999[dof], (pos, stat)


def two_token_pair(alpha):
    """(p, q) logits over two tokens with sum_x min(p, q) = alpha."""
    gap = 1.0 - alpha
    a = 0.5 + gap / 2
    b = 0.5 - gap / 2
    return np.log([a, 1 - a]), np.log([b, 1 - b])


def simulate_accepted(alphas, rows):
    k = len(alphas)
    pairs = [two_token_pair(a) for a in alphas]
    P = np.stack([pp for pp, _ in pairs] + [pairs[-1][0]]).astype(np.float32)
    Q = np.stack([qq for _, qq in pairs]).astype(np.float32)
    P = np.tile(P, (rows, 1, 1))
    Q = np.tile(Q, (rows, 1, 1))
    drafts = draft_from_oracle(Q, seed=1, offset=0)
    res = verify.spec_verify(P, Q, drafts, seed=0, offset=0)
    return np.array([r["accepted"] for r in res], dtype=np.float64)


@pytest.mark.slow
def test_expected_accepted_exercise_39_3(golden):
    g = golden("expected_accepted.json")["exercise_39_3"]
    acc = simulate_accepted(g["alpha"], rows=12000)
    se = acc.std() / math.sqrt(acc.size)
    assert abs(acc.mean() - g["expected_accepted"]) < 4 * se


@pytest.mark.slow
def test_expected_tokens_closed_form(golden):
    g = golden("expected_accepted.json")["equal_alpha"]
    emitted = simulate_accepted([g["alpha"]] * g["K"], rows=8000) + 1.0
    se = emitted.std() / math.sqrt(emitted.size)
    assert abs(emitted.mean() - g["expected_tokens"]) < 4 * se


def test_identical_draft_accepts_everything():
    rng = np.random.default_rng(10)
    z = rng.normal(0, 2, size=(4, 50)).astype(np.float32)
    P = np.stack([z] * 6)                 # [B=6, K+1=4, V]
    Q = P[:, :3].copy()
    drafts = draft_from_oracle(Q, seed=1, offset=0)
    res = verify.spec_verify(P, Q, drafts, seed=0, offset=0)
    assert all(r["accepted"] == 3 for r in res)
    assert all(r["ids"][:3] == list(drafts[r["row"]]) for r in res)


# ------------------------------------------------------------------ error rows

def test_error_rows():
    z = np.array([np.nan, -np.inf, np.nan])
    assert sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 0, 0.5)["status"] == sampler.ROW_NONFINITE
    assert sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 1, 0.5)["token"] == -1
    z = np.array([0.0, np.inf])
    assert sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 0, 0.5)["status"] == sampler.ROW_NONFINITE
    z = np.array([0.0, 1.0, np.nan])
    assert sampler.sample_row(z, -1.0, 0, 1.0, 0.0, 0, 0.5)["status"] == sampler.ROW_BAD_PARAMS
    assert sampler.sample_row(z, 1.0, -3, 1.0, 0.0, 0, 0.5)["status"] == sampler.ROW_BAD_PARAMS
    assert sampler.sample_row(z, 1.0, 0, float("nan"), 0.0, 0, 0.5)["status"] == sampler.ROW_BAD_PARAMS
    assert sampler.sample_row(z, 1.0, 0, 1.0, -0.1, 0, 0.5)["status"] == sampler.ROW_BAD_PARAMS
    ok = sampler.sample_row(z, 1.0, 0, 1.0, 0.0, 0, 0.999)
    assert ok["status"] == sampler.ROW_OK and ok["token"] == 1       # NaN counts as -inf
    P = np.zeros((1, 2, 4), dtype=np.float32)
    Q = np.zeros((1, 1, 4), dtype=np.float32)
    out = verify.spec_verify(P, Q, np.array([[4]]), 0, 0)[0]
    assert out["accepted"] == -1 and out["ids"] == [-1, -1]
    Q[0, 0, :] = np.nan
    out = verify.spec_verify(P, Q, np.array([[1]]), 0, 0)[0]
    assert out["status"] == sampler.ROW_NONFINITE


def test_row_results_do_not_depend_on_batch_subset():
    batch = workloads.random_sampler_batch(12, 300, dtype="f32", seed=3)
    full = sampler.sample(batch.values, batch.params, 7, 2)
    part = sampler.sample(batch.values, batch.params, 7, 2, rows=[5, 9])
    assert [full[5]["token"], full[9]["token"]] == [part[0]["token"], part[1]["token"]]
    assert philox.uniform(7, 2, 5, 0) == full[5]["u"]
