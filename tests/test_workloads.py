"""The seeded input generators (no arithmetic of the method): shapes, seeds
and the structure the parity tests rely on."""

import numpy as np

from spec_verify_gb300 import workloads


def _allowed_counts(allowed, vocab):
    ids = np.arange(vocab)
    return [int(((row[ids // 32] >> (ids % 32).astype(np.uint32)) & 1).sum()) for row in allowed]


def test_prepass_inputs_structure():
    batch = workloads.random_sampler_batch(10, 1000, dtype="f32", seed=3)
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=4)
    assert allowed.shape == (10, (1000 + 31) // 32) and allowed.dtype == np.uint32
    assert history.shape == (10, 64) and history.dtype == np.int32
    assert penalty.shape == (10,) and penalty.dtype == np.float32
    counts = _allowed_counts(allowed, 1000)
    assert counts[0] == 1 and counts[-1] == 0            # one allowed token; none
    assert all(0 < c < 1000 for c in counts[1:-1])
    assert set(np.unique(penalty)) <= {np.float32(x) for x in (1.0, 1.1, 1.3, 2.0, 0.8)}
    for b in range(10):
        top = set(np.argsort(-batch.values[b], kind="stable")[:32])
        h = history[b]
        assert len(top & set(h.tolist())) >= 1             # the penalty can matter
        assert (h < 0).any() or (h >= 1000).any()           # padding present
        assert len(h[(h >= 0) & (h < 1000)]) > len(set(h[(h >= 0) & (h < 1000)].tolist()))   # repeats


def test_prepass_inputs_are_seeded():
    batch = workloads.random_sampler_batch(4, 300, dtype="bf16", seed=1)
    a = workloads.prepass_inputs(batch.values, seed=9)
    b = workloads.prepass_inputs(batch.values, seed=9)
    c = workloads.prepass_inputs(batch.values, seed=10)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[1], c[1])


def test_bf16_rounding_of_the_generators_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, np.inf, -np.inf], dtype=np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    back = workloads.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even gives 1
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0078125)
    assert back[3] == -2.5 and np.isinf(back[4]) and back[5] == -np.inf


def test_verify_workload_shapes():
    vb = workloads.verify_workload()
    assert vb.shape == (32, 4, 32000)
    assert vb.p.shape == (32, 5, 32000) and vb.q.shape == (32, 4, 32000)
    small = workloads.verify_workload(batch=3, k=2, vocab=17, dtype="bf16", seed_id=5)
    assert small.p.dtype == np.uint16 and small.values("p").dtype == np.float32
