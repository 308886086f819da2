"""The multi-process path of bench.py on CPU: two gloo ranks.

Rows are independent, so N GPUs split a batch by rows with no collective on
the data path: rank r takes a contiguous block of rows and passes the global
index of its first row as row_base, so the Philox counter of every row is its
global index and the tokens do not depend on the split.  What the ranks share
is the timing: every rank reports its time, the job takes as long as the
slowest rank, and the job's rate counts the rows of all ranks.  These tests
run that host logic with the gloo backend and the oracle standing in for the
device (no GPU needed).
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

WORLD = 2
ROWS = 10


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    from spec_verify_gb300 import workloads
    return workloads.random_sampler_batch(ROWS, 257, dtype="bf16", seed=7, kinds="mixed")


def _verify_batch():
    from oracle import sampler as osam
    from spec_verify_gb300 import workloads
    vb = workloads.verify_workload(batch=ROWS, k=3, vocab=300, seed_id=41)
    qv = vb.values("q")
    res = osam.sample(qv.reshape(ROWS * 3, 300), workloads.make_params(ROWS * 3), 1, 0)
    drafts = np.array([r["token"] for r in res], dtype=np.int32).reshape(ROWS, 3)
    return vb, drafts


def _rank_main(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from oracle import sampler as osam
        from oracle import verify as over

        lo, hi = bench.row_block(ROWS, rank, WORLD)
        # sampler: this rank's block of one shared batch, keyed by row_base
        batch = _batch()
        res = osam.sample(batch.values[lo:hi], batch.params[lo:hi], 3, 1, row_base=lo)
        ids = torch.full((ROWS,), -9, dtype=torch.int64)
        ids[lo:hi] = torch.tensor([r["token"] for r in res])
        # verifier: the same split
        vb, drafts = _verify_batch()
        vres = over.spec_verify(vb.values("p")[lo:hi], vb.values("q")[lo:hi], drafts[lo:hi], 3, 1, row_base=lo)
        vids = torch.full((ROWS, 4), -9, dtype=torch.int64)
        vids[lo:hi] = torch.tensor([r["ids"] for r in vres])
        gathered = [torch.zeros(ROWS, dtype=torch.int64) for _ in range(WORLD)]
        dist.all_gather(gathered, ids)
        vgathered = [torch.zeros(ROWS, 4, dtype=torch.int64) for _ in range(WORLD)]
        dist.all_gather(vgathered, vids)
        merged = torch.stack(gathered).max(dim=0).values
        vmerged = torch.stack(vgathered).max(dim=0).values
        fake_seconds = 0.5 + rank        # rank 1 is the slowest
        slowest = bench.max_over_ranks(fake_seconds)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([slowest, bench.job_rate(hi - lo, WORLD, slowest)] + merged.tolist()
                         + vmerged.view(-1).tolist(), dtype=np.float64))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_rows_like_one_process(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=WORLD, start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    # every rank sees the slowest rank's time and the same whole-job rate
    assert r0[0] == r1[0] == 1.5
    assert r0[1] == r1[1] == 2 * (ROWS // 2) / 1.5
    np.testing.assert_array_equal(r0[2:], r1[2:])
    # the gathered tokens equal one process's tokens on the whole batch
    from oracle import sampler as osam
    from oracle import verify as over
    batch = _batch()
    want = [r["token"] for r in osam.sample(batch.values, batch.params, 3, 1)]
    assert list(r0[2:2 + ROWS].astype(int)) == want
    vb, drafts = _verify_batch()
    vwant = [x for r in over.spec_verify(vb.values("p"), vb.values("q"), drafts, 3, 1) for x in r["ids"]]
    assert list(r0[2 + ROWS:].astype(int)) == vwant


def test_row_blocks_cover_the_batch_once():
    import bench
    for rows in (1, 7, 256, 1000):
        for world in (1, 2, 3, 8):
            blocks = [bench.row_block(rows, r, world) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == rows
            assert all(blocks[i][1] == blocks[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in blocks]
            assert max(sizes) - min(sizes) <= 1
