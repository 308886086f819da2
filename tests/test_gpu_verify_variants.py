"""CUDA verifier with per-row knobs (smp_spec_verify_params, through the C ABI)
against the fp64 oracle: temperature and filters on p and q ("Speculative
decoding -- Hinglish notes", section "Temperature and Sampling"; eq. 39.2 of
"Decoding & Speculative Sampling"), greedy verification ("Inference: Sampling,
the KV Cache, Speculative Decoding and int8", section "Speculative decoding"),
and rows whose knobs are invalid."""

import numpy as np
import pytest

from oracle import sampler as osam
from oracle import verify as over
from spec_verify_gb300 import binding, workloads
from tests.parity import compare_verify, device_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def drafts_from_q(q_values, temperatures, seed=1, offset=0):
    """Draft ids drawn from q at each batch row's temperature (oracle sampler)."""
    b, k, v = q_values.shape
    prm = workloads.make_params(b * k)
    prm["temperature"] = np.repeat(np.asarray(temperatures, dtype=np.float32), k)
    res = osam.sample(q_values.reshape(b * k, v), prm, seed, offset)
    return np.array([r["token"] for r in res], dtype=np.int32).reshape(b, k)


def run(p_data, q_data, dtype, drafts, params, seed, offset):
    p = device_logits(p_data, dtype)
    q = device_logits(q_data, dtype)
    d = torch.from_numpy(np.ascontiguousarray(drafts, dtype=np.int32)).cuda()
    acc, ids, status = binding.spec_verify_params(p, q, d, params, seed, offset)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), ids.cpu().numpy(), int(status.cpu()[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k,vocab", [(2, 64), (4, 4099), (5, 32000)])
def test_temperature_parity(dtype, k, vocab):
    batch = 24
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype=dtype, seed_id=200 + k)
    temps = np.array([0.5, 0.7, 0.9, 1.0, 1.3, 2.0], dtype=np.float32)[np.arange(batch) % 6]
    prm = workloads.make_params(batch)
    prm["temperature"] = temps
    drafts = drafts_from_q(vb.values("q"), temps)
    acc, ids, status = run(vb.p, vb.q, dtype, drafts, prm, 11, 3)
    assert status == 0
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 11, 3, params=prm)
    compare_verify(want, acc, ids).check()
    assert any(r["accepted"] < k for r in want) and any(r["accepted"] > 0 for r in want)


def test_unit_temperature_equals_the_plain_call():
    vb = workloads.verify_workload(batch=16, k=3, vocab=5000, dtype="bf16", seed_id=41)
    drafts = drafts_from_q(vb.values("q"), np.ones(16))
    p = device_logits(vb.p, "bf16")
    q = device_logits(vb.q, "bf16")
    d = torch.from_numpy(drafts).cuda()
    plain = binding.spec_verify(p, q, d, 5, 6)
    ones = binding.spec_verify_params(p, q, d, workloads.make_params(16), 5, 6)
    none = binding.spec_verify_params(p, q, d, None, 5, 6)
    torch.cuda.synchronize()
    for other in (ones, none):
        assert torch.equal(plain[0], other[0]) and torch.equal(plain[1], other[1])
        assert int(other[2].cpu()[0]) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [7, 1000, 32003])
def test_greedy_parity_and_target_greedy_decoding(dtype, vocab):
    batch, k = 20, 4
    rng = np.random.default_rng(300 + vocab)
    if vocab < 100:   # integer logits: many ties at the top
        p = rng.integers(-3, 3, (batch, k + 1, vocab)).astype(np.float32)
    else:
        p = rng.normal(0, 2, (batch, k + 1, vocab)).astype(np.float32)
    q = rng.normal(0, 2, (batch, k, vocab)).astype(np.float32)
    q[1::3] = np.nan   # greedy verification never reads q
    p_data = workloads.f32_to_bf16_bits(p) if dtype == "bf16" else p
    q_data = workloads.f32_to_bf16_bits(q) if dtype == "bf16" else q
    p_vals = workloads.bf16_bits_to_f32(p_data) if dtype == "bf16" else p
    q_vals = workloads.bf16_bits_to_f32(q_data) if dtype == "bf16" else q
    tops = np.argmax(p_vals, axis=2)   # the target's greedy tokens (lowest id on ties)
    drafts = tops[:, :k].astype(np.int32).copy()
    for r in range(batch):   # row r keeps r % (k + 1) drafts
        m = r % (k + 1)
        if m < k:
            drafts[r, m] = (tops[r, m] + 1 + r % (vocab - 1)) % vocab
    prm = workloads.make_params(batch)
    prm["greedy"][0::2] = 1
    prm["temperature"][1::2] = 0.0   # T == 0 is greedy too
    prm["top_k"][2::4] = 5           # other knobs are ignored by greedy rows
    acc, ids, status = run(p_data, q_data, dtype, drafts, prm, 0, 0)
    assert status == 0
    want = over.spec_verify(p_vals, q_vals, drafts, 0, 0, params=prm)
    compare_verify(want, acc, ids).check()
    for r in range(batch):
        m = r % (k + 1)
        assert acc[r] == m
        assert list(ids[r, : m + 1]) == list(tops[r, : m + 1])   # greedy decoding with the target
        assert np.all(ids[r, m + 1:] == -1)


def test_mixed_modes_and_bad_knobs():
    batch, k, vocab = 16, 3, 3001
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype="f32", seed_id=57)
    prm = workloads.make_params(batch)
    prm["temperature"][0:4] = [0.6, 1.0, 1.7, 0.8]
    prm["greedy"][4:7] = 1
    prm["temperature"][7] = -1.0
    prm["temperature"][8] = np.nan
    prm["temperature"][9] = np.inf
    prm["top_k"][10] = 40
    prm["top_p"][11] = 0.9
    prm["min_p"][12] = 0.05
    prm["top_k"][13] = vocab     # off: top_k >= V
    prm["min_p"][14] = 1.0       # off: min_p >= 1
    prm["top_k"][15] = -2        # invalid
    drafts = drafts_from_q(vb.values("q"), np.where(prm["temperature"] > 0, prm["temperature"], 1.0)
                           .astype(np.float32).clip(0.1, 10))
    acc, ids, status = run(vb.p, vb.q, "f32", drafts, prm, 21, 4)
    bad = [7, 8, 9, 15]   # rows 10..12 are filtered (drafts drawn without the filters)
    assert status == binding.ROW_BAD_PARAMS
    assert all(acc[r] == -1 and np.all(ids[r] == -1) for r in bad)
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 21, 4, params=prm)
    assert [r["status"] for r in want if r["row"] in bad] == [osam.ROW_BAD_PARAMS] * len(bad)
    compare_verify(want, acc, ids).check()


def test_greedy_error_rows():
    rng = np.random.default_rng(61)
    p = rng.normal(0, 1, (4, 3, 50)).astype(np.float32)
    q = rng.normal(0, 1, (4, 2, 50)).astype(np.float32)
    p[1, 2, :] = np.nan          # no finite target logit at position K
    drafts = np.array([[1, 2], [3, 4], [50, 5], [6, 7]], dtype=np.int32)   # row 2: id out of range
    prm = workloads.make_params(4, greedy=1)
    acc, ids, status = run(p, q, "f32", drafts, prm, 0, 0)
    assert list(acc[1:3]) == [-1, -1] and np.all(ids[1:3] == -1)
    assert status == (binding.ROW_NONFINITE | binding.ROW_BAD_DRAFT)
    want = over.spec_verify(p, q, drafts, 0, 0, params=prm, rows=[0, 3])
    compare_verify(want, acc, ids).check()


def test_temperature_verify_output_follows_target_chi_square():
    # the output at each position is distributed as softmax(p_logits / T)
    rng = np.random.default_rng(71)
    vocab, k, rows, t = 8, 2, 100_000, 0.6
    zp = rng.normal(0, 1.0, (k + 1, vocab)).astype(np.float32)
    zq = rng.normal(0, 1.0, (k, vocab)).astype(np.float32)
    P = np.ascontiguousarray(np.tile(zp, (rows, 1, 1)))
    Q = np.ascontiguousarray(np.tile(zq, (rows, 1, 1)))
    ql = torch.from_numpy(Q.reshape(rows * k, vocab)).cuda()
    d, _, _ = binding.sample(ql, workloads.make_params(rows * k, temperature=t), 1, 0)
    drafts = d.view(rows, k).cpu().numpy()
    acc, ids, status = run(P, Q, "f32", drafts, workloads.make_params(rows, temperature=t), 0, 0)
    assert status == 0
    for pos in range(k + 1):
        reached = acc >= pos
        counts = np.bincount(ids[reached, pos], minlength=vocab)
        target = over.softmax64(zp[pos], t) * reached.sum()
        stat = float(np.sum((counts - target) ** 2 / target))
        assert stat < 24.32, (pos, stat)   # chi-square, 7 degrees of freedom, p = 0.001


def drafts_from_filtered_q(q_values, prm):
    """Draft ids drawn from q~ with each batch row's knobs (oracle sampler)."""
    b, k, v = q_values.shape
    res = osam.sample(q_values.reshape(b * k, v), np.repeat(prm, k), 1, 0)
    return np.array([r["token"] for r in res], dtype=np.int32).reshape(b, k)


FILTER_KNOBS = [  # (temperature, top_k, top_p, min_p)
    (1.0, 5, 1.0, 0.0), (0.7, 40, 1.0, 0.0), (1.0, 0, 0.9, 0.0), (1.5, 0, 0.5, 0.0),
    (1.0, 0, 1.0, 0.05), (0.8, 0, 1.0, 0.2), (0.9, 40, 0.9, 0.05), (1.2, 100, 0.95, 0.02),
    (1.0, 0, 1.0, 0.0), (0.6, 1, 1.0, 0.0), (1.0, 0, 0.999, 0.0), (2.0, 3, 0.8, 0.1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k,vocab", [(3, 517), (4, 4099), (4, 32000)])
def test_filtered_parity(dtype, k, vocab):
    batch = 24
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype=dtype, seed_id=400 + vocab % 97 + k)
    prm = workloads.make_params(batch)
    for r in range(batch):
        t, tk, tp, mp = FILTER_KNOBS[r % len(FILTER_KNOBS)]
        prm[r] = (t, tk, tp, mp, 0)
    drafts = drafts_from_filtered_q(vb.values("q"), prm)
    acc, ids, status = run(vb.p, vb.q, dtype, drafts, prm, 13, 7)
    assert status == 0
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 13, 7, params=prm)
    compare_verify(want, acc, ids).check()
    assert any(r["accepted"] < k for r in want) and any(r["accepted"] > 0 for r in want)


def test_filtered_output_follows_filtered_target():
    # p = (.4, .3, .2, .1), q = (.3, .1, .4, .2), top_k = 2 on both: p~ = (4/7, 3/7, 0, 0),
    # q~ = (3/7, 0, 4/7, 0); mean accepted length sum min(p~, q~) = 3/7 (K = 1), and
    # both emitted positions follow p~.
    rows = 200_000
    zp = np.log([0.4, 0.3, 0.2, 0.1]).astype(np.float32)
    zq = np.log([0.3, 0.1, 0.4, 0.2]).astype(np.float32)
    P = np.ascontiguousarray(np.tile(np.stack([zp, zp]), (rows, 1, 1)))
    Q = np.ascontiguousarray(np.tile(zq[None], (rows, 1, 1)))
    prm = workloads.make_params(rows, top_k=2)
    ql = torch.from_numpy(Q.reshape(rows, 4)).cuda()
    d, _, _ = binding.sample(ql, prm, 1, 0)
    drafts = d.view(rows, 1).cpu().numpy()
    assert set(np.unique(drafts)) == {0, 2}
    acc, ids, status = run(P, Q, "f32", drafts, prm, 0, 0)
    assert status == 0
    alpha = 3 / 7
    assert abs(acc.mean() - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / rows)
    p_tilde = np.array([4 / 7, 3 / 7, 0, 0])
    for pos in (0, 1):
        reached = acc >= pos
        counts = np.bincount(ids[reached, pos], minlength=4)
        assert counts[2] == 0 and counts[3] == 0
        target = p_tilde[:2] * reached.sum()
        stat = float(np.sum((counts[:2] - target) ** 2 / target))
        assert stat < 10.83, (pos, stat)   # chi-square, 1 degree of freedom, p = 0.001


ALPHA_ATOL = 1e-5   # binary32 probabilities (Z within about 1e-6 relative), exact fixed-point sums


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k,vocab", [(2, 300), (4, 32000)])
def test_acceptance_rates_parity(dtype, k, vocab):
    batch = 24
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype=dtype, seed_id=500 + k)
    prm = workloads.make_params(batch)
    for r in range(batch):
        t, tk, tp, mp = FILTER_KNOBS[r % len(FILTER_KNOBS)]
        prm[r] = (t, tk, tp, mp, 0)
    prm["greedy"][5] = 1            # alpha undefined: NaN
    prm["temperature"][7] = -1.0    # error row: NaN
    drafts = drafts_from_filtered_q(vb.values("q"), prm)   # row 7 gets draft -1: its knobs are invalid anyway
    p = device_logits(vb.p, dtype)
    q = device_logits(vb.q, dtype)
    d = torch.from_numpy(drafts).cuda()
    alpha = torch.full((batch, k), -7.0, dtype=torch.float32, device="cuda")
    acc, ids, status = binding.spec_verify_params(p, q, d, prm, 3, 1, out_alpha=alpha)
    torch.cuda.synchronize()
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 3, 1, params=prm, alpha=True)
    compare_verify(want, acc.cpu().numpy(), ids.cpu().numpy()).check()
    got = alpha.cpu().numpy()
    for r in want:
        w = np.array(r["alpha"])
        if np.all(np.isnan(w)):
            assert np.all(np.isnan(got[r["row"]])), r["row"]
        else:
            np.testing.assert_allclose(got[r["row"]], w, rtol=0, atol=ALPHA_ATOL, err_msg=str(r["row"]))
    assert int(status.cpu()[0]) == binding.ROW_BAD_PARAMS


def test_acceptance_rates_without_knobs_and_the_unchanged_draw():
    # out_alpha with no knobs: alpha at T = 1; the accepted lengths and ids are
    # those of the plain call
    vb = workloads.verify_workload(batch=16, k=3, vocab=5003, dtype="f32", seed_id=61)
    drafts = drafts_from_q(vb.values("q"), np.ones(16))
    p = device_logits(vb.p, "f32")
    q = device_logits(vb.q, "f32")
    d = torch.from_numpy(drafts).cuda()
    alpha = torch.empty((16, 3), dtype=torch.float32, device="cuda")
    plain = binding.spec_verify(p, q, d, 9, 2)
    withalpha = binding.spec_verify_params(p, q, d, None, 9, 2, out_alpha=alpha)
    torch.cuda.synchronize()
    assert torch.equal(plain[0], withalpha[0]) and torch.equal(plain[1], withalpha[1])
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 9, 2, alpha=True)
    np.testing.assert_allclose(alpha.cpu().numpy(), np.array([r["alpha"] for r in want]), rtol=0,
                               atol=ALPHA_ATOL)
