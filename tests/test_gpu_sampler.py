"""CUDA sampler (through the C ABI) against the fp64 oracle."""

import math
import os
import zlib

import numpy as np
import pytest

from oracle import pool as opool
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


def run(batch, seed=None, offset=None):
    logits = device_logits(batch.data, batch.dtype)
    ids, probs, status = binding.sample(logits, batch.params,
                                        batch.seed if seed is None else seed,
                                        batch.offset if offset is None else offset)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), probs.cpu().numpy(), int(status.cpu()[0])


def oracle(batch, rows=None, seed=None, offset=None):
    return osam.sample(batch.values, batch.params, batch.seed if seed is None else seed,
                       batch.offset if offset is None else offset, rows=rows)


# ------------------------------------------------------------------ the named workloads at full size

@pytest.mark.parametrize("name", ["basic", "mixed", "large_vocab", "flat_nucleus"])
def test_workload_parity(name):
    # Every row of every named workload, in the launch configuration the
    # bench times; the oracle runs on all host cores for the large batches.
    batch = workloads.sampler_workload(name)
    ids, probs, status = run(batch)
    assert status == 0
    if batch.data.size > 10**6:
        want = opool.sample_parallel(batch.values, batch.params, batch.seed, batch.offset)
    else:
        want = oracle(batch)
    assert len(want) == batch.data.shape[0]
    verdict = compare_sampler(want, ids, probs)
    verdict.check()
    assert verdict.compared == batch.data.shape[0] and not verdict.excused


# ------------------------------------------------------------------ a batch split by rows

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_row_base_split_equals_whole(dtype):
    # Rows are independent and the Philox counter holds the global row index
    # row_base + b, so two calls on the halves of a batch, each with the index
    # of its first row, give exactly the tokens of one call on the whole.
    batch = workloads.random_sampler_batch(40, 3001, dtype=dtype, seed=31, kinds="mixed")
    logits = device_logits(batch.data, batch.dtype)
    whole_ids, whole_probs, st = binding.sample(logits, batch.params, 5, 2)
    parts = []
    for lo, hi in ((0, 17), (17, 40)):
        ids, probs, st2 = binding.sample_rows(logits[lo:hi].contiguous(), batch.params[lo:hi], 5, 2, row_base=lo)
        parts.append((ids, probs, st2))
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and all(int(p[2].item()) == 0 for p in parts)
    assert torch.equal(torch.cat([p[0] for p in parts]), whole_ids)
    assert torch.equal(torch.cat([p[1] for p in parts]), whole_probs)
    # and the oracle with the same row bases agrees
    want = oracle(batch, seed=5, offset=2)
    compare_sampler(want, whole_ids.cpu().numpy(), whole_probs.cpu().numpy()).check()
    half = osam.sample(batch.values[17:], batch.params[17:], 5, 2, row_base=17)
    assert [r["token"] for r in half] == [r["token"] for r in want[17:]]


# ------------------------------------------------------------------ small seeded batches, ragged vocabularies

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kinds", ["mixed", "greedy", "minp", "topk", "topp", "plain"])
def test_random_parity(dtype, kinds):
    batch = workloads.random_sampler_batch(24, 10007, dtype=dtype, seed=zlib.crc32(f"{dtype}/{kinds}".encode()) % 1000,
                                           kinds=kinds)
    ids, probs, status = run(batch, seed=11, offset=3)
    assert status == 0
    compare_sampler(oracle(batch, seed=11, offset=3), ids, probs).check()


@pytest.mark.parametrize("vocab", [1, 2, 7, 33, 1000, 4099, 65537])
def test_vocab_sizes(vocab):
    batch = workloads.random_sampler_batch(9, vocab, dtype="bf16", seed=vocab, kinds="mixed")
    ids, probs, status = run(batch)
    assert status == 0
    compare_sampler(oracle(batch), ids, probs).check()


def test_filter_debug_matches_eq_39_2():
    batch = workloads.random_sampler_batch(16, 5003, dtype="bf16", seed=5, kinds="mixed")
    logits = device_logits(batch.data, batch.dtype)
    ids, probs, full, kept, status = binding.filter_debug(logits, batch.params, 0, 0)
    torch.cuda.synchronize()
    full = full.cpu().numpy()
    kept = kept.cpu().numpy()
    want = osam.filtered_rows(batch.values, batch.params)
    for b, (pt, size) in enumerate(want):
        assert kept[b] == size, b
        assert np.array_equal(full[b] > 0, pt > 0) or np.array_equal(full[b] != 0, pt != 0), b
        nz = pt > 0
        np.testing.assert_allclose(full[b][nz], pt[nz], rtol=PROB_RTOL, atol=0)


# ------------------------------------------------------------------ edge cases

def make_batch(rows, params, dtype="f32"):
    data = np.asarray(rows, dtype=np.float32)
    if dtype == "bf16":
        data = workloads.f32_to_bf16_bits(data)
    return workloads.Batch("edge", dtype, data, params)


def test_ties_split_by_top_k_and_top_p():
    # 4000 tokens on 5 distinct values: top-k and top-p boundaries fall inside
    # tie buckets and must take the lower ids first.
    rng = np.random.default_rng(1)
    rows = rng.choice([0.0, -0.5, -1.0, -2.0, -3.0], size=(12, 4000)).astype(np.float32)
    prm = workloads.make_params(12)
    prm["top_k"][:6] = [1, 7, 100, 1000, 2500, 3999]
    prm["top_p"][6:] = [0.01, 0.2, 0.5, 0.7, 0.9, 0.999]
    for dtype in ("f32", "bf16"):
        batch = make_batch(rows, prm, dtype)
        ids, probs, _ = run(batch, seed=4)
        compare_sampler(oracle(batch, seed=4), ids, probs).check()
        logits = device_logits(batch.data, dtype)
        _, _, full, kept, _ = binding.filter_debug(logits, prm, 4, 0)
        kept = kept.cpu().numpy()
        want = osam.filtered_rows(batch.values, prm)
        assert [k for _, k in want] == list(kept)
        full = full.cpu().numpy()
        for b, (pt, _) in enumerate(want):
            assert np.array_equal(full[b] > 0, pt > 0), b


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("vocab", [33, 40, 100, 130, 257, 1000])
def test_top_k_near_vocab_on_short_rows(vocab, dtype):
    # k above the number of lanes that hold data in a row's first batch: the
    # streaming lower bound of the k-th value is then -inf, and the padding
    # past the end of the batch must still never become a candidate.
    rng = np.random.default_rng(vocab)
    rows = rng.normal(0.0, 2.0, size=(8, vocab)).astype(np.float32)
    prm = workloads.make_params(8)
    prm["top_k"] = [min(vocab - 1, 128), vocab - 1, vocab // 2, 64, 5, 2, 1, 100]
    batch = make_batch(rows, prm, dtype)
    ids, probs, status = run(batch, seed=9)
    assert status == 0
    assert ids.min() >= 0 and ids.max() < vocab
    compare_sampler(oracle(batch, seed=9), ids, probs).check()
    logits = device_logits(batch.data, dtype)
    _, _, full, kept, _ = binding.filter_debug(logits, prm, 9, 0)
    want = osam.filtered_rows(batch.values, prm)
    assert [k for _, k in want] == list(kept.cpu().numpy())
    full = full.cpu().numpy()
    for b, (pt, _) in enumerate(want):
        np.testing.assert_allclose(full[b], pt, rtol=PROB_RTOL, atol=1e-7)


def test_error_rows_and_flags():
    V = 64
    rows = np.random.default_rng(2).normal(0, 1, size=(8, V)).astype(np.float32)
    rows[0, :] = np.nan
    rows[1, :] = -np.inf
    rows[2, 5] = np.inf
    rows[3, ::2] = np.nan                       # NaN counts as -inf, row still valid
    prm = workloads.make_params(8)
    prm["temperature"][4] = -1.0
    prm["top_k"][5] = -2
    prm["top_p"][6] = np.nan
    prm["min_p"][7] = -0.5
    batch = make_batch(rows, prm)
    ids, probs, status = run(batch)
    want = oracle(batch)
    assert [r["token"] for r in want] == list(ids)
    assert ids[3] >= 0 and ids[3] % 2 == 1
    assert status == (binding.ROW_NONFINITE | binding.ROW_BAD_PARAMS)
    assert all(math.isnan(p) for p in probs[[0, 1, 2, 4, 5, 6, 7]])


def test_greedy_and_zero_temperature_lowest_id():
    rows = np.zeros((3, 300), dtype=np.float32)
    rows[:, [17, 120, 250]] = 5.0
    prm = workloads.make_params(3, temperature=1.0)
    prm["greedy"][0] = 1
    prm["temperature"][1] = 0.0
    prm["temperature"][2] = 1e-3                # sampling, but effectively the tied top tokens
    ids, probs, _ = run(make_batch(rows, prm))
    assert ids[0] == 17 and ids[1] == 17 and probs[0] == 1.0
    assert ids[2] in (17, 120, 250)


def test_signed_zero_and_min_p_one():
    rows = np.array([[0.0, -0.0, -1.0, -0.0, 0.0]], dtype=np.float32)
    prm = workloads.make_params(1, greedy=1)
    ids, _, _ = run(make_batch(rows, prm))
    assert ids[0] == 0
    prm = workloads.make_params(1, min_p=1.0)   # min_p >= 1 is off
    batch = make_batch(rows, prm)
    ids, probs, _ = run(batch, seed=9)
    compare_sampler(oracle(batch, seed=9), ids, probs).check()


def test_misaligned_base_pointer():
    batch = workloads.random_sampler_batch(6, 3001, dtype="bf16", seed=12, kinds="mixed")
    big = np.zeros((6 * 3001 + 3,), dtype=np.uint16)
    big[3:] = batch.data.reshape(-1)
    t = torch.from_numpy(big.view(np.int16)).view(torch.bfloat16).cuda()
    logits = t[3:].view(6, 3001)                 # base 6 bytes past a 16-byte boundary
    ids, probs, status = binding.sample(logits, batch.params, 0, 0)
    torch.cuda.synchronize()
    compare_sampler(oracle(batch), ids.cpu().numpy(), probs.cpu().numpy()).check()


def test_more_rows_than_resident_ctas():
    # 700 rows on at most 2 CTAs per SM: CTAs take several rows, and the copy
    # cursor runs ahead across rows of both paths (general rows in between).
    batch = workloads.random_sampler_batch(700, 3001, dtype="bf16", seed=23, kinds="mixed")
    ids, probs, status = run(batch, seed=3, offset=1)
    assert status == 0
    rows = list(range(0, 700, 7)) + [699]
    compare_sampler(oracle(batch, rows=rows, seed=3, offset=1), ids, probs).check()


def test_repeatable_and_offset_changes_draws():
    batch = workloads.random_sampler_batch(32, 2000, dtype="f32", seed=3, kinds="plain")
    a = run(batch, seed=1, offset=0)
    b = run(batch, seed=1, offset=0)
    c = run(batch, seed=1, offset=1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[0], c[0])


def test_draw_histogram_chi_square():
    z = np.array([2.0, 1.0, 0.5, 0.0, -1.0, -3.0, -7.0, 1.5], dtype=np.float32)
    rows = 200_000
    prm = workloads.make_params(rows, temperature=0.9, top_k=6, top_p=0.97)
    logits = torch.from_numpy(np.tile(z, (rows, 1))).cuda()
    ids, _, status = binding.sample(logits, prm, 8, 0)
    counts = np.bincount(ids.cpu().numpy(), minlength=z.size)
    _, _, pt, _ = osam.filtered_distribution(z, 0.9, top_k=6, top_p=0.97)
    mask = pt > 0
    assert np.all(counts[~mask] == 0)
    expected = pt[mask] * rows
    stat = float(np.sum((counts[mask] - expected) ** 2 / expected))
    dof = int(mask.sum()) - 1
    assert stat < {3: 16.27, 4: 18.47, 5: 20.52}[dof]


def test_wait_expiry_marks_rows_and_the_next_call_is_correct(monkeypatch):
    # Every wait of the streamed sampler for a TMA batch is bounded.  With the
    # limit at 0 a wait gives up at the first poll that finds its batch
    # missing, which happens on a normal input: the CTA lets its copies in
    # flight land, gives the rows from that one on the id -1, sets
    # SMP_ROW_TIMEOUT and returns.  Rows finished before keep their tokens.
    batch = workloads.sampler_workload("large_vocab", batch=64)
    logits = device_logits(batch.data, batch.dtype)
    want = [r["token"] for r in oracle(batch)]
    monkeypatch.setenv("SMP_WAIT_LIMIT_NS", "0")
    flagged = 0
    for i in range(5):
        ids, probs, status = binding.sample(logits, batch.params, batch.seed, batch.offset)
        torch.cuda.synchronize()
        st = int(status.item())
        got = ids.cpu().numpy()
        assert st in (0, binding.ROW_TIMEOUT), st
        for b in range(64):
            assert got[b] == -1 or got[b] == want[b], (i, b, got[b], want[b])
        if st:
            flagged += 1
            assert (got == -1).any()
        else:
            assert (got == np.array(want)).all()
    assert flagged > 0
    monkeypatch.delenv("SMP_WAIT_LIMIT_NS")
    ids, probs, status = run(batch)
    assert status == 0
    compare_sampler(oracle(batch), ids, probs).check()
