"""CUDA beam-step candidate selection (smp_beam_topk, through the C ABI)
against the fp64 oracle ("Decoding & Speculative Sampling", section 39.1,
eq. 39.1, Listing 39.1)."""

import math

import numpy as np
import pytest

from oracle import beam as obeam
from spec_verify_gb300 import binding, workloads
from tests.parity import BAND, EXCUSE_FRACTION, device_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCORE_ATOL = 1e-5   # log Z from binary32 exponentials: within about 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def run(data, dtype, scores, width):
    logits = device_logits(data.reshape(-1, data.shape[-1]), dtype).view(*data.shape)
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float64)).cuda()
    parent, token, score, status = binding.beam_topk(logits, s, width)
    torch.cuda.synchronize()
    return parent.cpu().numpy(), token.cpu().numpy(), score.cpu().numpy(), int(status.cpu()[0])


def compare(want, parent, token, score, exact=False):
    excused, failed = [], []
    for r in want:
        g = r["group"]
        same = list(parent[g]) == r["parent"] and list(token[g]) == r["token"]
        if not same:
            (excused if (r["margin"] < BAND and not exact) else failed).append((g, r["margin"]))
            continue
        if r["status"] == obeam.GROUP_OK:
            w = np.array(r["score"])
            fin = np.isfinite(w)
            assert np.all(np.isfinite(score[g][fin]))
            np.testing.assert_allclose(score[g][fin], w[fin], rtol=0, atol=SCORE_ATOL)
            rest_w, rest_g = w[~fin], score[g][~fin]
            assert np.all((rest_w == rest_g) | (np.isnan(rest_w) & np.isnan(rest_g)))
        else:
            assert np.all(np.isnan(score[g]))
    assert not failed, failed[:8]
    assert len(excused) <= math.floor(EXCUSE_FRACTION * len(want)), excused[:8]


def beam_batch(groups, beams, vocab, dtype, seed):
    rng = np.random.default_rng(90_000 + seed)
    z = workloads.zipf_logits_f32(rng, groups * beams, vocab).reshape(groups, beams, vocab)
    scores = -rng.uniform(0, 12, (groups, beams))
    if dtype == "bf16":
        data = workloads.f32_to_bf16_bits(z)
        return data, workloads.bf16_bits_to_f32(data), scores
    return z, z, scores


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("beams,width,vocab", [(1, 1, 1000), (1, 5, 7), (2, 2, 4099), (4, 4, 32000),
                                               (4, 8, 32000), (8, 8, 50021), (16, 32, 3001), (3, 32, 5)])
def test_beam_parity(dtype, beams, width, vocab):
    data, values, scores = beam_batch(6, beams, vocab, dtype, seed=beams * 100 + width)
    if beams > 1:
        scores[2, 1] = -np.inf          # a dead beam
    parent, token, score, status = run(data, dtype, scores, width)
    assert status == 0
    want = obeam.beam_step(values, scores, width)
    compare(want, parent, token, score)


def test_infinities_and_nan_slices():
    # +inf anywhere makes the beam's row non-finite; a slice of only NaN or
    # -inf is not an error when the rest of the row is finite
    data, values, scores = beam_batch(3, 2, 20000, "f32", seed=9)
    data[0, 1, 17000] = np.inf
    data[1, 0, :9000] = np.nan
    data[2, 1, 5000:] = -np.inf
    values = data
    parent, token, score, status = run(data, "f32", scores, 2)
    assert status == binding.ROW_NONFINITE
    assert np.all(parent[0] == -1)
    want = obeam.beam_step(values, scores, 2, groups=[1, 2])
    compare(want, parent, token, score)


def test_fewer_finite_logits_than_width():
    # NaN counts as -inf: with fewer finite logits than the width, the rest
    # of the kept candidates score -inf in flat-index order
    z = np.full((2, 2, 3000), -np.inf, dtype=np.float32)
    z[:, :, 10] = 1.0
    z[:, 0, 20] = 0.5
    z[0, 1, 100:140] = np.nan
    scores = np.array([[0.0, -1.0], [-2.0, 0.0]])
    parent, token, score, status = run(z, "f32", scores, 6)
    assert status == 0
    want = obeam.beam_step(z, scores, 6)
    compare(want, parent, token, score, exact=True)


def test_flat_rows_take_the_radix_path():
    # every logit equal: all of a slice ties at the threshold, more than the
    # list holds, so the exact radix selection picks the lowest ids
    z = np.zeros((2, 3, 40000), dtype=np.float32)
    z[1, 2, 39999] = 0.25
    scores = np.array([[0.0, -0.5, -0.25], [-1.0, -1.0, -1.0]])
    parent, token, score, status = run(z, "f32", scores, 8)
    want = obeam.beam_step(z, scores, 8)
    compare(want, parent, token, score, exact=True)


def test_ties_within_a_beam_follow_the_flat_index():
    # one beam, integer logits: equal logits give equal scores by the same
    # formula on both sides, so the lower token id must come first, exactly
    rng = np.random.default_rng(5)
    z = rng.integers(-3, 3, (10, 1, 3000)).astype(np.float32)
    scores = np.zeros((10, 1))
    parent, token, score, status = run(z, "f32", scores, 32)
    want = obeam.beam_step(z, scores, 32)
    compare(want, parent, token, score, exact=True)


def test_error_groups():
    data, values, scores = beam_batch(4, 3, 500, "f32", seed=7)
    scores[1, 2] = np.nan
    data[2, 0, :] = np.nan
    parent, token, score, status = run(data, "f32", scores, 3)
    assert status == (binding.ROW_BAD_PARAMS | binding.ROW_NONFINITE)
    for g in (1, 2):
        assert np.all(parent[g] == -1) and np.all(token[g] == -1) and np.all(np.isnan(score[g]))
    want = obeam.beam_step(values, scores, 3, groups=[0, 3])
    compare(want, parent, token, score)


def test_two_step_search_example():
    # the page's example: a beam of two finds B then "end" at 0.36 > greedy's 0.24
    eps = 1e-12
    def logp(prefix):
        p = np.full(6, eps)
        if prefix == ():
            p[0], p[1] = 0.6, 0.4
        elif prefix == (0,):
            p[2], p[3], p[4] = 0.4, 0.3, 0.3
        else:
            p[5], p[3] = 0.9, 0.1
        return np.log(p / p.sum()).astype(np.float32)
    parent, token, score, _ = run(logp(())[None, None], "f32", np.zeros((1, 1)), 2)
    beams = [(int(t),) for t in token[0]]
    assert beams == [(0,), (1,)]
    z2 = np.stack([logp(b) for b in beams])[None]
    parent2, token2, score2, _ = run(z2, "f32", score, 2)
    best = beams[parent2[0, 0]] + (int(token2[0, 0]),)
    assert best == (1, 5) and abs(math.exp(score2[0, 0]) - 0.36) < 1e-6
