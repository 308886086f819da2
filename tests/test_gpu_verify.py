"""CUDA speculative verifier (through the C ABI) against the fp64 oracle."""

import numpy as np
import pytest

from oracle import pool as opool
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


def test_verify_parity_over_1e5_rows():
    # The verify workload's 32 batch rows verified as 3125 parts of a
    # 100,000-row batch (row bases 0, 32, 64, ...): the logits repeat, the
    # uniforms of every part are new.  At most 1e-4 of the rows may differ,
    # and only where the oracle's margin is inside the 1e-6 band.
    vb = workloads.verify_workload()
    B, K, V = vb.shape
    drafts = oracle_drafts(vb.values("q"), vb.draft_seed, vb.draft_offset)
    p = device_logits(vb.p, vb.dtype)
    q = device_logits(vb.q, vb.dtype)
    d = torch.from_numpy(drafts).cuda()
    tiles = 3125
    ws = torch.zeros(binding.spec_verify_workspace_bytes(B, K), dtype=torch.uint8, device="cuda")
    acc = torch.empty(tiles, B, dtype=torch.int32, device="cuda")
    ids = torch.empty(tiles, B, K + 1, dtype=torch.int32, device="cuda")
    status = torch.empty(tiles, dtype=torch.int32, device="cuda")
    for t in range(tiles):
        binding.spec_verify_rows(p, q, d, None, vb.seed, vb.offset, row_base=t * B, workspace=ws,
                                 out_accepted=acc[t], out_ids=ids[t], status=status[t:t + 1])
    torch.cuda.synchronize()
    assert int(status.abs().max().item()) == 0
    want = opool.spec_verify_tiled(vb.values("p"), vb.values("q"), drafts, vb.seed, vb.offset,
                                   [t * B for t in range(tiles)])
    for r in want:
        r["row"] = r["row_base"] + r["row"]
    verdict = compare_verify(want, acc.view(-1).cpu().numpy(), ids.view(-1, K + 1).cpu().numpy())
    verdict.check()
    assert verdict.compared == tiles * B


def test_verify_row_base_split_equals_whole():
    vb = workloads.verify_workload(batch=24, k=3, vocab=4099, dtype="bf16", seed_id=211)
    drafts = oracle_drafts(vb.values("q"), 1, 0)
    p = device_logits(vb.p, vb.dtype)
    q = device_logits(vb.q, vb.dtype)
    d = torch.from_numpy(drafts).cuda()
    prm = workloads.make_params(24, temperature=0.9)
    prm["top_p"][::3] = 0.9
    prm["greedy"][5] = 1
    whole = binding.spec_verify_params(p, q, d, prm, 3, 4)
    parts = [binding.spec_verify_rows(p[lo:hi].contiguous(), q[lo:hi].contiguous(), d[lo:hi].contiguous(),
                                      prm[lo:hi], 3, 4, row_base=lo) for lo, hi in ((0, 10), (10, 24))]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([x[0] for x in parts]), whole[0])
    assert torch.equal(torch.cat([x[1] for x in parts]), whole[1])
    want = over.spec_verify(vb.values("p")[10:], vb.values("q")[10:], drafts[10:], 3, 4, params=prm[10:],
                            row_base=10)
    for r in want:
        r["row"] += 10
    compare_verify(want, whole[0].cpu().numpy(), whole[1].cpu().numpy()).check()


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


def test_exact_accept_retest_gives_the_same_results(monkeypatch):
    # An accept test whose two sides lie within the fast Z's error bound is
    # decided again on Z recomputed exactly; SMP_VERIFY_EXACT_ACCEPT sends
    # every test down that path.  Both paths must give the oracle's results,
    # and the same ones wherever the fast path was certain (everywhere here).
    for dtype, k, vocab, seed_id in (("f32", 4, 32000, 17), ("bf16", 3, 4099, 18)):
        vb = workloads.verify_workload(batch=16, k=k, vocab=vocab, dtype=dtype, seed_id=seed_id)
        drafts = oracle_drafts(vb.values("q"), 1, 0)
        fast = run_verify(vb.p, vb.q, dtype, drafts, 2, 5)
        monkeypatch.setenv("SMP_VERIFY_EXACT_ACCEPT", "1")
        exact = run_verify(vb.p, vb.q, dtype, drafts, 2, 5)
        monkeypatch.delenv("SMP_VERIFY_EXACT_ACCEPT")
        assert fast[2] == exact[2] == 0
        assert np.array_equal(fast[0], exact[0]) and np.array_equal(fast[1], exact[1])
        want = over.spec_verify(vb.values("p"), vb.values("q"), drafts, 2, 5)
        compare_verify(want, exact[0], exact[1]).check()
