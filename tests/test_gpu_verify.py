"""CUDA speculative verifier (through the C ABI) against the fp64 oracle."""

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


def oracle_drafts(q_values, seed, offset):
    b, k, v = q_values.shape
    res = osam.sample(q_values.reshape(b * k, v), workloads.make_params(b * k), seed, offset)
    return np.array([r["token"] for r in res], dtype=np.int32).reshape(b, k)


def run_verify(p_data, q_data, dtype, drafts, seed, offset):
    p = device_logits(p_data, dtype)
    q = device_logits(q_data, dtype)
    d = torch.from_numpy(np.ascontiguousarray(drafts, dtype=np.int32)).cuda()
    acc, ids, status = binding.spec_verify(p, q, d, seed, offset)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), ids.cpu().numpy(), int(status.cpu()[0])


def test_verify_workload_parity():
    vb = workloads.verify_workload()
    drafts = oracle_drafts(vb.values("q"), vb.draft_seed, vb.draft_offset)
    acc, ids, status = run_verify(vb.p, vb.q, vb.dtype, drafts, vb.seed, vb.offset)
    assert status == 0
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, vb.seed, vb.offset)
    compare_verify(want, acc, ids).check()
    # both paths (rejection and bonus) are exercised by this workload
    assert any(r["accepted"] < 4 for r in want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k,vocab", [(1, 8), (3, 1000), (5, 4099), (16, 257)])
def test_verify_random_parity(dtype, k, vocab):
    vb = workloads.verify_workload(batch=16, k=k, vocab=vocab, dtype=dtype, seed_id=100 + k)
    drafts = oracle_drafts(vb.values("q"), 1, 0)
    acc, ids, status = run_verify(vb.p, vb.q, dtype, drafts, 7, 2)
    assert status == 0
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 7, 2)
    compare_verify(want, acc, ids).check()


def test_identical_draft_accepts_all():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 2, size=(8, 5, 300)).astype(np.float32)
    q = np.ascontiguousarray(z[:, :4])
    drafts = oracle_drafts(q, 1, 0)
    acc, ids, status = run_verify(z, q, "f32", drafts, 0, 0)
    assert np.all(acc == 4)
    assert np.array_equal(ids[:, :4], drafts)
    want = over.spec_verify(z, q, drafts, 0, 0)
    compare_verify(want, acc, ids).check()


def test_verify_error_rows():
    rng = np.random.default_rng(4)
    p = rng.normal(0, 1, size=(4, 3, 50)).astype(np.float32)
    q = rng.normal(0, 1, size=(4, 2, 50)).astype(np.float32)
    drafts = np.array([[1, 2], [50, 3], [4, -1], [5, 6]], dtype=np.int32)
    q[3, 1, :] = np.nan
    acc, ids, status = run_verify(p, q, "f32", drafts, 0, 0)
    assert list(acc[1:]) == [-1, -1, -1]
    assert np.all(ids[1:] == -1)
    assert status == (binding.ROW_BAD_DRAFT | binding.ROW_NONFINITE)
    want = over.spec_verify(p, q, drafts, 0, 0, rows=[0])
    compare_verify(want, acc, ids).check()


def test_verify_output_follows_target_chi_square():
    rng = np.random.default_rng(9)
    vocab, k, rows = 8, 2, 100_000
    zp = rng.normal(0, 1.5, size=(k + 1, vocab)).astype(np.float32)
    zq = rng.normal(0, 1.5, size=(k, vocab)).astype(np.float32)
    P = np.ascontiguousarray(np.tile(zp, (rows, 1, 1)))
    Q = np.ascontiguousarray(np.tile(zq, (rows, 1, 1)))
    # drafts from q with the CUDA sampler (T = 1, no filters), seed 1
    ql = torch.from_numpy(Q.reshape(rows * k, vocab)).cuda()
    d, _, _ = binding.sample(ql, workloads.make_params(rows * k), 1, 0)
    drafts = d.view(rows, k).cpu().numpy()
    acc, ids, status = run_verify(P, Q, "f32", drafts, 0, 0)
    assert status == 0
    crit = {7: 24.32}
    for pos in range(k + 1):
        reached = acc >= pos
        counts = np.bincount(ids[reached, pos], minlength=vocab)
        target = over.softmax64(zp[pos]) * reached.sum()
        stat = float(np.sum((counts - target) ** 2 / target))
        assert stat < crit[vocab - 1], (pos, stat)


def test_verify_results_do_not_depend_on_cluster_size(monkeypatch):
    vb = workloads.verify_workload(batch=12, k=3, vocab=5003, dtype="f32", seed_id=31)
    drafts = oracle_drafts(vb.values("q"), 1, 0)
    outs = []
    for cluster in ("1", "2", "4", "8"):
        monkeypatch.setenv("SMP_FORCE_CLUSTER", cluster)
        outs.append(run_verify(vb.p, vb.q, vb.dtype, drafts, 4, 9))
    monkeypatch.delenv("SMP_FORCE_CLUSTER")
    for acc, ids, status in outs:
        assert status == 0
        assert np.array_equal(acc, outs[0][0])
        assert np.array_equal(ids, outs[0][1])
    want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 4, 9)
    compare_verify(want, outs[0][0], outs[0][1]).check()
