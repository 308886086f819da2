"""Pins of the logit pre-pass oracle: the repetition penalty ("Choosing the
next word", section "The repetition penalty") and the constraint mask
("Decoding & Speculative Sampling", section 39.3, Listing 39.3).

Each pin rests on what the pages or the mathematics fix:
* the penalty's two branches on hand values, and that both lower the score
  for r > 1 (the page says so);
* a masked softmax is the model's distribution conditioned on the allowed set
  (section 39.3), computed here the other way round: full softmax, then
  renormalised over the allowed set;
* the tiny JSON-number grammar of Listing 39.3 drives the mask: after '['
  only digits come out, after a digit only ']' or ',', and an empty allowed
  set is an invalid state (error row);
* bf16 rounding against numpy's float32 view of known bit patterns.
"""

import math

import numpy as np
import pytest

from oracle import prepass
from oracle import sampler as osam


def test_penalty_branches_on_hand_values():
    assert prepass.penalize(2.0, 2.0) == np.float32(1.0)
    assert prepass.penalize(-1.0, 2.0) == np.float32(-2.0)
    assert prepass.penalize(0.0, 1.5) == np.float32(0.0)       # z <= 0 branch: 0 * r
    assert prepass.penalize(3.0, 1.0) == np.float32(3.0)
    assert prepass.penalize(1.0, 3.0) == np.float32(1.0) / np.float32(3.0)   # binary32 division


def test_penalty_lowers_every_score_for_r_above_one():
    rng = np.random.default_rng(1)
    z = rng.normal(0, 4, 2000).astype(np.float32)
    for r in (1.1, 1.5, 2.0):
        out = np.array([prepass.penalize(v, r) for v in z])
        nz = z != 0
        assert np.all(out[nz] < z[nz])
        assert np.all(out[~nz] == 0)


def test_round_to_bf16_known_patterns():
    cases = {0x3F800000: 0x3F800000,   # 1.0 exact
             0x3F808000: 0x3F800000,   # halfway, even below: down
             0x3F818000: 0x3F820000,   # halfway, odd below: up
             0x3F808001: 0x3F810000,   # above halfway: up
             0xBF80FFFF: 0xBF810000,   # negative, rounds away in magnitude
             0x7F7FFFFF: 0x7F800000}   # the largest float rounds to infinity
    for src, want in cases.items():
        x = np.array(src, dtype=np.uint32).view(np.float32)[()]
        got = np.array(prepass.round_to_bf16(x), dtype=np.float32).view(np.uint32)[()]
        assert int(got) == want, hex(src)
    assert math.isnan(prepass.round_to_bf16(np.float32(np.nan)))


def test_history_penalises_each_distinct_token_once():
    z = np.array([2.0, -1.0, 0.5, 4.0], dtype=np.float32)
    once = prepass.prepare_row(z, history=[3], penalty=2.0)
    many = prepass.prepare_row(z, history=[3, 3, -1, 3, 99], penalty=2.0)
    assert np.array_equal(once, many)
    assert list(once) == [2.0, -1.0, 0.5, 2.0]
    both = prepass.prepare_row(z, history=[1, 0], penalty=2.0)
    assert list(both) == [1.0, -2.0, 0.5, 4.0]


def _words(allowed):
    allowed = np.asarray(allowed, dtype=bool)
    n = (allowed.size + 31) // 32
    words = np.zeros(n, dtype=np.uint32)
    for i in np.flatnonzero(allowed):
        words[i // 32] |= np.uint32(1) << np.uint32(i % 32)
    return words


def test_masked_distribution_is_conditioned_on_the_allowed_set():
    rng = np.random.default_rng(2)
    v = 70
    z = rng.normal(0, 2, v).astype(np.float32)
    allowed = rng.random(v) < 0.4
    zm = prepass.prepare_row(z, allowed_words=_words(allowed))
    p_masked = osam.softmax_with_temperature(osam.logits_to_f64(zm), 1.0)
    p = osam.softmax_with_temperature(z.astype(np.float64), 1.0)
    conditioned = np.where(allowed, p, 0.0) / np.sum(p[allowed])
    np.testing.assert_allclose(p_masked, conditioned, rtol=1e-12, atol=1e-300)


VOCAB = ["[", "]", ","] + [str(d) for d in range(10)] + ["a"]


def grammar_allowed(prefix):
    """Listing 39.3's tiny grammar '[' digit (',' digit)* ']', restated."""
    if not prefix:
        return np.array([t == "[" for t in VOCAB])
    if prefix[-1] in {"[", ","}:
        return np.array([t.isdigit() for t in VOCAB])
    if prefix[-1].isdigit():
        return np.array([t in {"]", ","} for t in VOCAB])
    return np.zeros(len(VOCAB), dtype=bool)


@pytest.mark.parametrize("prefix", ["", "[", "[7", "[7,", "[7,3]", "[3", "[3,"])   # Exercise 39.4's prefixes too
def test_tiny_grammar_mask(prefix):
    from spec_verify_gb300 import workloads
    rows = 300
    rng = np.random.default_rng(3)
    logits = rng.normal(0, 2, (rows, len(VOCAB))).astype(np.float32)
    allowed = grammar_allowed(prefix)
    words = np.tile(_words(allowed), (rows, 1))
    prm = workloads.make_params(rows, temperature=1.3)
    prm["greedy"][::3] = 1
    res = prepass.sample_processed(logits, prm, 4, 0, allowed=words)
    if not allowed.any():
        assert all(r["token"] == -1 and r["status"] == osam.ROW_NONFINITE for r in res)
        return
    toks = [r["token"] for r in res]
    assert all(allowed[t] for t in toks)
    assert len(set(toks)) > 1 or allowed.sum() == 1


def test_penalty_and_mask_order_and_bad_penalty():
    from spec_verify_gb300 import workloads
    z = np.array([[1.0, 0.9, -5.0, 0.2]], dtype=np.float32)
    prm = workloads.make_params(1, greedy=1)
    hist = np.array([[0, -1]])
    # the penalty moves the arg-max from token 0 to token 1
    assert prepass.sample_processed(z, prm, 0, 0, history=hist, penalty=np.array([1.2]))[0]["token"] == 1
    # masking token 1 as well leaves token 0, penalised, against tokens 2 and 3
    words = np.array([[0b1101]], dtype=np.uint32)
    assert prepass.sample_processed(z, prm, 0, 0, allowed=words, history=hist,
                                    penalty=np.array([1.2]))[0]["token"] == 0
    assert prepass.sample_processed(z, prm, 0, 0, allowed=words, history=hist,
                                    penalty=np.array([20.0]))[0]["token"] == 3
    for bad in (0.0, -1.0, np.nan, np.inf):
        r = prepass.sample_processed(z, prm, 0, 0, history=hist, penalty=np.array([bad]))[0]
        assert r["token"] == -1 and r["status"] == osam.ROW_BAD_PARAMS


@pytest.mark.parametrize("prefix, allowed_tokens", [
    ("[", set("0123456789")), ("[3", {"]", ","}), ("[3,", set("0123456789")), ("", {"["}),
])
def test_exercise_39_4_allowed_next_tokens(prefix, allowed_tokens):
    # "Decoding & Speculative Sampling", Exercise 39.4: the grammar [ d (, d)* ]
    # allows these next tokens after each prefix
    got = {VOCAB[i] for i in np.flatnonzero(grammar_allowed(prefix))}
    assert got == allowed_tokens
