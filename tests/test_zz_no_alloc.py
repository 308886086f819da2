"""smp_spec_verify_static: the verifier for callers that cannot allocate.

Callers inside an allocator or memory-pool callback, runtimes that forbid
cudaMalloc once serving, or loops that must not let an allocation synchronise
the device cannot hand the verifier a workspace.  smp_spec_verify_static uses
a fixed device array owned by the library instead.  These tests call it
through the C ABI and check that it returns exactly what smp_spec_verify
returns with a caller workspace, on two calls in a row (the second call finds
the first call's data still in the shared array).  This file is named so that
pytest collects it last.
"""

import ctypes

import numpy as np
import pytest

from oracle import sampler as osam
from spec_verify_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def inputs(batch, k, vocab, dtype, seed_id):
    vb = workloads.verify_workload(batch=batch, k=k, vocab=vocab, dtype=dtype, seed_id=seed_id)
    qv = vb.values("q")
    res = osam.sample(qv.reshape(batch * k, vocab), workloads.make_params(batch * k), 1, 0)
    drafts = np.array([r["token"] for r in res], dtype=np.int32).reshape(batch, k)

    def up(a):
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    return up(vb.p), up(vb.q), torch.from_numpy(drafts).cuda()


def call_static(p, q, d, seed, offset):
    """smp_spec_verify_static through ctypes, outputs preallocated here."""
    lib = binding.load()
    batch, k1, vocab = p.shape
    acc = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    ids = torch.full((batch, k1), -7, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    dtype = binding.SMP_BF16 if p.dtype == torch.bfloat16 else binding.SMP_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.smp_spec_verify_static(ctypes.c_void_p(p.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(d.data_ptr()), batch, k1 - 1, vocab, dtype, seed,
                                    offset, ctypes.c_void_p(acc.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                    ctypes.c_void_p(status.data_ptr()), stream)
    assert rc == 0, lib.smp_status_string(rc)
    return acc, ids, status


def test_static_scratch_matches_workspace_twice_in_a_row():
    cases = [(32, 4, 32000, "f32", 5, 0, 0), (48, 6, 5003, "bf16", 6, 3, 9)]
    for batch, k, vocab, dtype, seed_id, seed, offset in cases:
        p, q, d = inputs(batch, k, vocab, dtype, seed_id)
        acc_s, ids_s, st_s = call_static(p, q, d, seed, offset)
        acc_w, ids_w, st_w = binding.spec_verify(p, q, d, seed, offset)
        torch.cuda.synchronize()
        assert torch.equal(acc_s, acc_w)
        assert torch.equal(ids_s, ids_w)
        assert int(st_s.item()) == int(st_w.item()) == 0
        assert int(acc_s.min().item()) >= 0


def test_static_rejects_batches_beyond_the_array():
    lib = binding.load()
    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    # 4096 rows with k = 16 need 4096 * 33 * 32 bytes, more than the 1 MiB array
    assert binding.spec_verify_workspace_bytes(4096, 16) > binding.STATIC_VERIFY_SCRATCH_BYTES
    rc = lib.smp_spec_verify_static(fake, fake, fake, 4096, 16, 1000, binding.SMP_F32, 0, 0, fake, fake,
                                    null, null)
    assert rc == 5   # SMP_ERR_WORKSPACE
    rc = lib.smp_spec_verify_static(fake, fake, fake, 8, 0, 1000, binding.SMP_F32, 0, 0, fake, fake, null, null)
    assert rc == 1   # SMP_ERR_INVALID_ARG
