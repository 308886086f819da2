"""The kept set of rows with top-k up to 128 and top-p (or min-p) from a ranked
candidate list, on the sampler's general path (binary32 rows; bf16 rows there
take the count table and are compared alike) and the verifier's filtered
rows of both types, against the fp64 oracle: candidates above the k-th largest thread
maximum, exact ranks by (logit desc, id asc), top-p decided from a bracket on
Z or, when a prefix lands inside it, from the exact Z; the draw read from the
list.  Rows with long runs of equal logits overflow the list and take the
radix selection.  Selection is "Decoding & Speculative Sampling", section 39.2
and eq. 39.2; the draw is "Choosing the next word", section "Where the
randomness comes from, and where it stops"."""

import numpy as np
import pytest

from oracle import prepass
from oracle import sampler as osam
from oracle import verify as over
from spec_verify_gb300 import binding, workloads
from tests.parity import PROB_RTOL, compare_sampler, compare_verify, device_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def batch_of(rows, prm, dtype):
    rows = np.asarray(rows, dtype=np.float32)
    data = workloads.f32_to_bf16_bits(rows) if dtype == "bf16" else np.ascontiguousarray(rows)
    return workloads.Batch("topk-list", dtype, data, prm)


def check(batch, seeds=((0, 0), (7, 3), (11, 9), (5, 1))):
    logits = device_logits(batch.data, batch.dtype)
    for seed, offset in seeds:
        ids, probs, status = binding.sample(logits, batch.params, seed, offset)
        torch.cuda.synchronize()
        want = osam.sample(batch.values, batch.params, seed, offset)
        compare_sampler(want, ids.cpu().numpy(), probs.cpu().numpy()).check()
    _, _, full, kept, _ = binding.filter_debug(logits, batch.params, 0, 0)
    torch.cuda.synchronize()
    want = osam.filtered_rows(batch.values, batch.params)
    assert [k for _, k in want] == list(kept.cpu().numpy())
    full = full.cpu().numpy()
    for b, (pt, _) in enumerate(want):
        np.testing.assert_allclose(full[b], pt, rtol=PROB_RTOL, atol=1e-9, err_msg=f"row {b}")


def knobs(n, top_k, top_p, min_p=0.0, temperature=1.0):
    prm = workloads.make_params(n, temperature=temperature)
    prm["top_k"] = top_k
    prm["top_p"] = top_p
    prm["min_p"] = min_p
    return prm


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [131, 4099, 32000])
def test_random_rows(dtype, vocab):
    rng = np.random.default_rng(vocab + (7 if dtype == "bf16" else 0))
    n = 16
    rows = rng.normal(0.0, 2.0, size=(n, vocab)).astype(np.float32)
    rows[8:] = workloads.zipf_logits_f32(rng, n - 8, vocab)
    k = np.array([1, 2, 7, 40, 100, 128, 50, 128] * 2, dtype=np.int32)
    prm = knobs(n, k, np.resize(np.float32([0.9, 0.5, 0.95, 0.99, 0.3, 0.999, 0.8, 0.9]), n),
                temperature=np.resize(np.float32([1.0, 0.7, 1.3, 0.5]), n))
    prm["min_p"][3::4] = 0.05
    check(batch_of(rows, prm, dtype))


def test_prefix_exactly_at_the_top_p_target():
    # a few equal maxima and -inf elsewhere: a prefix of j of them holds
    # exactly j / n of Z, so top_p = j / n sits on the target and inside the
    # bracket; the exact Z decides (the crossing counts as reached)
    V = 5003
    rows = np.full((8, V), -np.inf, dtype=np.float32)
    rows[0, [10, 20]] = 1.0
    rows[1, [3, 4, 5, 6]] = 0.0
    rows[2, [3, 4, 5, 6]] = 0.0
    rows[3, 100:108] = 2.5
    rows[4, [7, 9]] = 3.0
    rows[4, 50:60] = -40.0            # tiny masses that move Z by less than the bracket
    rows[5, :8] = 1.0
    rows[6, :3] = 0.0
    rows[7, [1, 2]] = 0.5
    prm = knobs(8, np.int32([5, 10, 10, 20, 6, 100, 3, 2]),
                np.float32([0.5, 0.75, 0.25, 0.375, 0.5, 0.625, 1.0 / 3.0, 0.5]))
    for dtype in ("f32", "bf16"):
        check(batch_of(rows, prm, dtype))


def test_ties_overflow_the_list_and_short_tie_rows_do_not():
    # every logit equal: with V > 1024 the candidates overflow and the radix
    # selection takes the row; with V <= 1024 the list holds the whole row and
    # ranks the ties by id
    rng = np.random.default_rng(3)
    big = np.zeros((4, 6007), dtype=np.float32)
    big[2] = rng.choice([1.0, 0.0], size=6007)
    big[3, ::2] = 0.5
    small = np.zeros((4, 900), dtype=np.float32)
    small[1] = rng.choice([1.0, 0.0, -1.0], size=900)
    for rows in (big, small):
        prm = knobs(4, np.int32([40, 128, 64, 3]), np.float32([0.9, 0.5, 0.99, 0.7]))
        check(batch_of(rows, prm, "f32"))
        check(batch_of(rows, prm, "bf16"))


def test_min_p_cuts_inside_the_first_k():
    rng = np.random.default_rng(17)
    rows = workloads.zipf_logits_f32(rng, 8, 12011)
    prm = knobs(8, np.int32([128, 100, 40, 128, 10, 128, 64, 2]),
                np.float32([0.99, 0.95, 0.9, 0.999, 0.5, 0.97, 0.9, 0.9]),
                min_p=np.float32([0.0, 0.01, 0.05, 0.1, 0.3, 1e-6, 0.5, 0.02]), temperature=0.9)
    check(batch_of(rows, prm, "bf16"))
    check(batch_of(rows, prm, "f32"))


def test_non_finite_logits_and_short_rows():
    rng = np.random.default_rng(29)
    V = 3001
    rows = rng.normal(0.0, 1.0, size=(6, V)).astype(np.float32)
    rows[0, ::5] = np.nan
    rows[1, 3:] = -np.inf               # three finite tokens, top-k past them
    rows[2, :V - 1] = -np.inf           # one finite token
    rows[3, 1000:2000] = np.nan
    rows[4, ::2] = -np.inf
    prm = knobs(6, np.int32([20, 10, 128, 128, 64, 5]), np.float32(0.9))
    check(batch_of(rows, prm, "f32"))
    short = rng.normal(0.0, 1.0, size=(4, 5)).astype(np.float32)
    check(batch_of(short, knobs(4, np.int32([1, 2, 3, 4]), np.float32([0.9, 0.5, 0.99, 0.3])), "f32"))


def test_misaligned_bf16_rows():
    rng = np.random.default_rng(41)
    V = 9999                            # odd: rows start off a 16-byte boundary
    rows = rng.normal(0.0, 1.5, size=(7, V)).astype(np.float32)
    rows[:, :3] = 5.0
    rows[:, -2:] = 5.5
    prm = knobs(7, np.int32([2, 3, 5, 40, 128, 1, 7]), np.float32([0.6, 0.9, 0.99, 0.95, 0.5, 0.9, 0.999]))
    check(batch_of(rows, prm, "bf16"), seeds=[(s, 0) for s in range(6)])


def test_pre_pass_rows():
    batch = workloads.random_sampler_batch(16, 12011, dtype="bf16", seed=71, kinds="topp")
    batch.params["top_k"] = np.resize(np.int32([40, 128, 7, 100]), 16)
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=72)
    logits = device_logits(batch.data, "bf16")
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
    for seed, offset in ((5, 2), (8, 1)):
        ids, probs, status = binding.sample_processed(logits, batch.params, seed, offset, to(allowed, np.int32),
                                                      to(history, np.int32), to(penalty, np.float32))
        torch.cuda.synchronize()
        want = prepass.sample_processed(batch.values, batch.params, seed, offset, dtype="bf16", allowed=allowed,
                                        history=history, penalty=penalty)
        compare_sampler(want, ids.cpu().numpy(), probs.cpu().numpy()).check()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verifier_rows_with_top_k(dtype):
    # the verifier's filtered rows: top-k with top-p and min-p on p and q
    batch, k, vocab = 16, 4, 32000
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype=dtype, seed_id=900 + (dtype == "bf16"))
    prm = workloads.make_params(batch)
    table = [(0.8, 40, 0.9, 0.0), (1.0, 1, 0.5, 0.0), (0.7, 128, 0.99, 0.0), (1.2, 2, 0.3, 0.0),
             (1.0, 64, 1.0, 0.1), (0.9, 100, 0.95, 0.02), (1.0, 7, 0.8, 0.0), (0.6, 128, 0.5, 0.0)]
    for r in range(batch):
        t, tk, tp, mp = table[r % len(table)]
        prm[r] = (t, tk, tp, mp, 0)
    res = osam.sample(vb.values("q").reshape(batch * k, vocab), np.repeat(prm, k), 1, 0)
    drafts = np.array([r["token"] for r in res], dtype=np.int32).reshape(batch, k)
    p = device_logits(vb.p, dtype)
    q = device_logits(vb.q, dtype)
    d = torch.from_numpy(drafts).cuda()
    acc, ids, status = binding.spec_verify_params(p, q, d, prm, 21, 4)
    torch.cuda.synchronize()
    assert int(status.cpu()[0]) == 0
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 21, 4, params=prm)
    compare_verify(want, acc.cpu().numpy(), ids.cpu().numpy()).check()


def test_top_p_within_a_few_millionths_of_a_prefix():
    # top_p placed 1.05e-6 to 1.3e-6 (of Z) from the mass of a prefix that
    # holds 70 to 97 % of it: outside the parity band, inside the binary32
    # bracket on Z (about 2e-6 of top_p * Z here), so these rows decide top-p
    # with the exact Z
    rng = np.random.default_rng(77)
    n, V = 48, 5003
    rows = rng.normal(0.0, 4.0, size=(n, V)).astype(np.float32)
    prm = knobs(n, np.int32(100), np.float32(0.9))
    deltas = np.array([-1.3e-6, -1.15e-6, -1.05e-6, 1.05e-6, 1.15e-6, 1.3e-6])
    for b in range(n):
        z = rows[b].astype(np.float64)
        order = np.lexsort((np.arange(V), -z))
        w = np.exp(z[order] - z.max())
        cum = np.cumsum(w) / w.sum()
        r = min(int(np.searchsorted(cum, rng.uniform(0.7, 0.97))) + 1, 99)
        prm["top_p"][b] = np.float32(cum[r - 1] + deltas[b % len(deltas)])
    prm["min_p"][::7] = 1e-4
    check(batch_of(rows, prm, "f32"))
