"""The multi-process path of bench.py on CPU: two gloo ranks.

Rows are independent, so N GPUs run N independent batches (weak scaling, no
collective on the data path).  What the ranks share is the timing: every rank
reports its time, the job takes as long as the slowest rank, and the job's
rate counts the rows of all ranks.  These tests run that host logic with the
gloo backend and the oracle standing in for the device (no GPU needed).
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from oracle import sampler as osam
        from spec_verify_gb300 import workloads

        # each rank samples its own batch, as bench.py does (seed = rank)
        batch = workloads.random_sampler_batch(6, 257, dtype="bf16", seed=7, kinds="mixed")
        res = osam.sample(batch.values, batch.params, rank, 0)
        ids = np.array([r["token"] for r in res], dtype=np.int64)
        fake_seconds = 0.5 + rank        # rank 1 is the slowest
        slowest = bench.max_over_ranks(fake_seconds)
        gathered = [torch.zeros(6, dtype=torch.int64) for _ in range(WORLD)]
        dist.all_gather(gathered, torch.from_numpy(ids))
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([slowest, bench.job_rate(6, WORLD, slowest)] +
                         [float(x) for t in gathered for x in t.tolist()]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_independent_rows(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=WORLD, start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    # every rank sees the slowest rank's time and the same whole-job rate
    assert r0[0] == r1[0] == 1.5
    assert r0[1] == r1[1] == 2 * 6 / 1.5
    # each rank's rows match the single-process oracle for its own seed
    from oracle import sampler as osam
    from spec_verify_gb300 import workloads
    batch = workloads.random_sampler_batch(6, 257, dtype="bf16", seed=7, kinds="mixed")
    for rank in range(WORLD):
        want = [r["token"] for r in osam.sample(batch.values, batch.params, rank, 0)]
        assert list(r0[2 + 6 * rank: 8 + 6 * rank].astype(int)) == want
    np.testing.assert_array_equal(r0[2:], r1[2:])
