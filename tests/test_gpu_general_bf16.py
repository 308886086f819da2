"""The sampler's general path on bf16 rows (per-value counts over a window of
binades, listed small magnitudes, the draw walked from either end) against
the fp64 oracle, on rows built to reach each of its cases: small-magnitude
tokens kept, dropped or too many for the list; a boundary among them; windows
on one side of zero; tokens below the window; a maximum past the window's
anchor; ties at the boundary drawn from both ends; min-p with top-p; extreme
temperatures; NaN and -inf; and the logit pre-pass.  Every row is a top-p or
plain-sampling row, so every row takes the general path (rows the table
cannot take fall back to the per-element path, which must agree as well).
Selection is "Decoding & Speculative Sampling", section 39.2 and eq. 39.2;
the draw is "Choosing the next word", section "Where the randomness comes
from, and where it stops"."""

import numpy as np
import pytest

from oracle import prepass
from oracle import sampler as osam
from spec_verify_gb300 import binding, workloads
from tests.parity import PROB_RTOL, compare_sampler, device_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def bf16_batch(rows, prm):
    data = workloads.f32_to_bf16_bits(np.asarray(rows, dtype=np.float32))
    return workloads.Batch("general-bf16", "bf16", data, prm)


def check(batch, seeds=((0, 0), (7, 3), (11, 9))):
    """Tokens and probabilities for several (seed, offset) pairs, so that the
    draws fall in both halves of Z_S; kept counts and p~ from the debug call."""
    logits = device_logits(batch.data, "bf16")
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


def top_p_params(n, top_p=0.95, temperature=1.0):
    prm = workloads.make_params(n, temperature=temperature)
    prm["top_p"] = top_p
    return prm


def test_small_magnitudes_listed_kept_and_overflowing():
    # near-flat rows (the window crosses zero) with exact zeros of both signs,
    # subnormals and tiny values: a few are listed one by one and kept; 300
    # overflow the list (the per-element path takes the row)
    rng = np.random.default_rng(101)
    V = 20011
    rows = rng.normal(0.0, 0.3, size=(8, V)).astype(np.float32)
    tiny = np.array([0.0, -0.0, 2.0 ** -130, -(2.0 ** -128), 2.0 ** -20, -(2.0 ** -17)], dtype=np.float32)
    for b, n in enumerate([0, 3, 40, 250, 300, 1000, 40, 40]):
        pos = rng.choice(V, size=n, replace=False)
        rows[b, pos] = rng.choice(tiny, size=n)
    prm = top_p_params(8)
    prm["top_p"][6] = 1.0          # plain sampling
    prm["top_p"][7] = 0.999
    check(bf16_batch(rows, prm))


def test_boundary_among_small_magnitudes():
    # half the mass on a few large logits, the rest on values within 2^-20 of
    # zero: a top-p crossing lands among the listed tokens
    V = 4099
    rows = np.full((4, V), -30.0, dtype=np.float32)
    rows[:, :4] = 2.0
    rng = np.random.default_rng(5)
    rows[:, 100:160] = rng.choice([0.0, -0.0, 2.0 ** -22, -(2.0 ** -21), 2.0 ** -25], size=(4, 60))
    prm = top_p_params(4)
    prm["top_p"] = [0.9, 0.5, 0.3, 0.999]
    check(bf16_batch(rows, prm))


@pytest.mark.parametrize("center", [60.0, -60.0, 33.5, -7.9])
def test_window_on_one_side_of_zero(center):
    # every logit far from zero: the window holds only positive (or only
    # negative) binades; 33.5 puts its bottom just above zero
    rng = np.random.default_rng(int(abs(center) * 10))
    rows = (center + rng.normal(0.0, 0.5, size=(6, 7001))).astype(np.float32)
    prm = top_p_params(6, top_p=0.9)
    prm["top_p"][3:] = [0.5, 0.99, 1.0]
    check(bf16_batch(rows, prm))


def test_tokens_below_the_window_and_top_k_past_them():
    # logits spread over [-120, 8]: most tokens lie below the window and have
    # zero mass; top-k past the window's tokens keeps k, the rest draw alike
    rng = np.random.default_rng(9)
    V = 9001
    rows = rng.uniform(-120.0, 8.0, size=(6, V)).astype(np.float32)
    prm = top_p_params(6, top_p=0.97)
    prm["top_k"] = [0, V - 5, 3000, 100, 10, 0]
    prm["top_p"][5] = 1.0
    check(bf16_batch(rows, prm))


def test_maximum_past_the_first_rounds():
    # the first round of the row anchors the window; a later maximum within
    # 8 T of it stays in the window, one further above it does not (the
    # per-element path takes that row)
    rng = np.random.default_rng(3)
    V = 40009
    rows = rng.normal(0.0, 0.3, size=(6, V)).astype(np.float32)
    rows[0, 30000] = 5.0
    rows[1, 39999] = 9.5
    rows[2, 20000] = 30.0
    rows[3, [25000, 25001, 25002]] = 2.5
    rows[4, V - 1] = 7.0
    prm = top_p_params(6, top_p=0.9)
    prm["temperature"][5] = 0.5
    check(bf16_batch(rows, prm))


def test_ties_at_the_boundary_from_both_ends():
    # five values, thousands of tokens each: the boundary value is cut inside
    # its ties (the first n tokens in id order are kept), and the draws walk
    # from both ends of the row
    rng = np.random.default_rng(21)
    rows = rng.choice([1.0, 0.5, 0.0, -0.5, -1.0], size=(16, 12289)).astype(np.float32)
    prm = top_p_params(16)
    prm["top_p"] = np.linspace(0.05, 0.99, 16).astype(np.float32)
    prm["top_k"][::5] = [17, 4000, 9000, 12000]
    seeds = [(s, o) for s in (1, 2, 3) for o in (0, 5)]
    check(bf16_batch(rows, prm), seeds=seeds)


def test_min_p_with_top_p():
    rng = np.random.default_rng(33)
    rows = workloads.zipf_logits_f32(rng, 8, 15013)
    prm = top_p_params(8, top_p=0.95, temperature=0.9)
    prm["min_p"] = [0.0, 0.01, 0.05, 0.1, 0.3, 1e-6, 0.5, 0.02]
    check(bf16_batch(rows, prm))


@pytest.mark.parametrize("temperature", [0.02, 0.3, 4.0, 25.0])
def test_extreme_temperatures(temperature):
    # a narrow window (low T) or one spanning many binades (high T, the list
    # bound g rises and more tokens are listed)
    rng = np.random.default_rng(int(temperature * 100))
    rows = workloads.zipf_logits_f32(rng, 6, 10007)
    rows[3] = rng.normal(0.0, 1.0, size=10007)
    prm = top_p_params(6, top_p=0.9, temperature=temperature)
    prm["top_p"][4:] = [1.0, 0.999]
    check(bf16_batch(rows, prm))


def test_nan_and_negative_infinity_in_general_rows():
    rng = np.random.default_rng(44)
    V = 6007
    rows = rng.normal(0.0, 1.0, size=(5, V)).astype(np.float32)
    rows[0, ::7] = np.nan
    rows[1, ::3] = -np.inf
    rows[2, :V - 2] = -np.inf          # two finite tokens
    rows[3, 1:] = np.nan               # one finite token
    rows[4, 100:200] = np.nan
    check(bf16_batch(rows, top_p_params(5, top_p=0.8)))


def test_misaligned_rows_with_odd_vocabulary():
    rng = np.random.default_rng(55)
    V = 9999                           # odd: every other row starts 2 bytes past a 16-byte boundary
    rows = rng.normal(0.0, 0.4, size=(7, V)).astype(np.float32)
    rows[:, :5] = 3.0                  # mass in the head edge
    rows[:, -3:] = 3.5                 # and in the tail edge
    prm = top_p_params(7, top_p=0.6)
    prm["top_p"][4:] = [0.01, 0.999, 1.0]
    check(bf16_batch(rows, prm), seeds=[(s, 0) for s in range(6)])


def test_pre_pass_on_general_rows():
    batch = workloads.random_sampler_batch(16, 12011, dtype="bf16", seed=61, kinds="topp")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=62)
    logits = device_logits(batch.data, "bf16")
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
    for seed, offset in ((5, 2), (8, 1)):
        ids, probs, status = binding.sample_processed(logits, batch.params, seed, offset, to(allowed, np.int32),
                                                      to(history, np.int32), to(penalty, np.float32))
        torch.cuda.synchronize()
        want = prepass.sample_processed(batch.values, batch.params, seed, offset, dtype="bf16", allowed=allowed,
                                        history=history, penalty=penalty)
        compare_sampler(want, ids.cpu().numpy(), probs.cpu().numpy()).check()
