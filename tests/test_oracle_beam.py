"""Pins of the beam-step oracle ("Decoding & Speculative Sampling", section
39.1, eq. 39.1, Listing 39.1; "Efficient Inference & Compression", section
"Beam search").

* the page's two-step example (A 0.6 / B 0.4; after A three tokens at 0.4,
  0.3, 0.3; after B "end" at 0.9): greedy ends at probability 0.24, a beam of
  two finds B-end at 0.36 -- run through the oracle's single step twice;
* brute force: the kept candidates are the first `width` of all beams x V
  candidates sorted by (score desc, flat index asc), with log p from
  scipy.special.log_softmax;
* width 1 from one beam of score 0 is greedy decoding (the arg-max, lowest
  id on ties);
* scores add: the kept scores are beam score + log p exactly (eq. 39.1).
"""

import math

import numpy as np
import pytest

from oracle import beam


def test_two_step_example_beats_greedy():
    # tokens: 0 = A, 1 = B, 2 = "continue", 3 = x, 4 = y, 5 = "end"
    eps = 1e-12
    def probs_after(prefix):
        p = np.full(6, eps)
        if prefix == ():
            p[0], p[1] = 0.6, 0.4
        elif prefix == (0,):
            p[2], p[3], p[4] = 0.4, 0.3, 0.3
        elif prefix == (1,):
            p[5] = 0.9
            p[3] = 0.1
        return np.log(p / p.sum())
    # step 1: one beam (the prompt), width 2
    s1 = beam.select_group(probs_after(())[None], np.array([0.0]), 2)
    beams = [(int(t),) for t in s1["token"]]
    assert beams == [(0,), (1,)]
    # step 2: both beams, width 2
    logits = np.stack([probs_after(b) for b in beams])
    s2 = beam.select_group(logits, np.array(s1["score"]), 2)
    best = (beams[s2["parent"][0]] + (s2["token"][0],), math.exp(s2["score"][0]))
    assert best[0] == (1, 5)
    assert abs(best[1] - 0.36) < 1e-9
    greedy = 0.6 * 0.4
    assert best[1] > greedy


def test_brute_force_against_log_softmax():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(1)
    for trial in range(20):
        W, V = rng.integers(1, 5), rng.integers(2, 30)
        z = rng.integers(-3, 4, (W, V)).astype(np.float32)          # ties everywhere
        s = rng.choice([0.0, -1.0, -2.5], size=W)
        width = int(rng.integers(1, W * V + 1))
        lp = special.log_softmax(z.astype(np.float64), axis=1) + s[:, None]
        flat = lp.ravel()
        order = sorted(range(flat.size), key=lambda i: (-flat[i], i))[:width]
        got = beam.select_group(z, s, width)
        assert got["parent"] == [i // V for i in order]
        assert got["token"] == [i % V for i in order]
        np.testing.assert_allclose(got["score"], flat[order], rtol=0, atol=1e-12)


def test_width_one_single_beam_is_greedy():
    rng = np.random.default_rng(2)
    for _ in range(30):
        z = rng.integers(-2, 3, 17).astype(np.float32)
        got = beam.select_group(z[None], np.array([0.0]), 1)
        assert got["parent"] == [0] and got["token"] == [int(np.argmax(z))]


def test_scores_add_and_dead_beams():
    z = np.array([[0.0, 1.0, 2.0], [2.0, 1.0, 0.0]], dtype=np.float32)
    s = np.array([-1.0, -np.inf])
    got = beam.select_group(z, s, 4)
    lp = beam.log_softmax64(z[0])
    assert got["parent"][:3] == [0, 0, 0] and got["token"][:3] == [2, 1, 0]
    np.testing.assert_allclose(got["score"][:3], -1.0 + lp[[2, 1, 0]], rtol=0, atol=0)
    assert got["parent"][3] == 1 and got["token"][3] == 0 and got["score"][3] == -np.inf


def test_error_groups():
    z = np.zeros((2, 5), dtype=np.float32)
    assert beam.select_group(z, np.array([0.0, np.nan]), 2)["status"] == beam.GROUP_BAD_SCORE
    z[1] = -np.inf
    r = beam.select_group(z, np.array([0.0, 0.0]), 2)
    assert r["status"] == beam.GROUP_NONFINITE and r["token"] == [-1, -1]


def test_width_past_the_candidates():
    z = np.array([[0.0, 1.0]], dtype=np.float32)
    got = beam.select_group(z, np.array([0.0]), 4)
    assert got["token"] == [1, 0, -1, -1] and got["parent"] == [0, 0, -1, -1]
    assert math.isnan(got["score"][2]) and math.isnan(got["score"][3])
