"""CUDA sampler with the logit pre-pass (smp_sample_processed, through the C
ABI) against the fp64 oracle: repetition penalty ("Choosing the next word",
section "The repetition penalty") and constraint mask ("Decoding &
Speculative Sampling", section 39.3)."""

import numpy as np
import pytest

from oracle import prepass
from oracle import sampler as osam
from spec_verify_gb300 import binding, workloads
from tests.parity import compare_sampler, device_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def run(batch, allowed, history, penalty, seed=5, offset=2):
    logits = device_logits(batch.data, batch.dtype)
    to = lambda a, dt: None if a is None else torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
    ids, probs, status = binding.sample_processed(logits, batch.params, seed, offset, to(allowed, np.int32),
                                                  to(history, np.int32), to(penalty, np.float32))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), probs.cpu().numpy(), int(status.cpu()[0])


def expected_status(results):
    st = 0
    for r in results:
        st |= r["status"]
    return st


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [1000, 32000, 50021])
@pytest.mark.parametrize("parts", ["both", "mask", "penalty"])
def test_prepass_parity(dtype, vocab, parts):
    batch = workloads.random_sampler_batch(24, vocab, dtype=dtype, seed=vocab % 89, kinds="mixed")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=vocab % 13)
    if parts == "mask":
        history = penalty = None
    if parts == "penalty":
        allowed = None
    ids, probs, status = run(batch, allowed, history, penalty)
    want = prepass.sample_processed(batch.values, batch.params, 5, 2, dtype=dtype, allowed=allowed,
                                    history=history, penalty=penalty)
    compare_sampler(want, ids, probs).check()
    assert status == expected_status(want)
    if parts != "penalty":
        assert want[-1]["status"] == osam.ROW_NONFINITE          # the row with no allowed token


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sparse_mask_with_top_k(dtype):
    # a grammar-like mask (a handful of allowed tokens) under top-k 40 and
    # min-p: fewer finite logits than k, so the masked tokens pad the top k
    batch = workloads.random_sampler_batch(16, 32000, dtype=dtype, seed=77, kinds="topk")
    batch.params["top_k"] = 40
    batch.params["min_p"][::2] = 0.05
    rng = np.random.default_rng(78)
    words = (32000 + 31) // 32
    allowed = np.zeros((16, words), dtype=np.uint32)
    for b in range(16):
        ids = rng.choice(32000, size=1 + b, replace=False)
        np.bitwise_or.at(allowed[b], ids // 32, (np.uint32(1) << (ids % 32).astype(np.uint32)))
    ids, probs, status = run(batch, allowed, None, None)
    want = prepass.sample_processed(batch.values, batch.params, 5, 2, dtype=dtype, allowed=allowed)
    compare_sampler(want, ids, probs).check()
    assert status == 0


def test_bad_penalty_rows():
    batch = workloads.random_sampler_batch(6, 700, dtype="f32", seed=3, kinds="mixed")
    _, history, _ = workloads.prepass_inputs(batch.values, seed=4)
    penalty = np.array([1.2, 0.0, -1.0, np.nan, np.inf, 1.0], dtype=np.float32)
    batch.params["greedy"][1] = 1    # greedy rows need a valid penalty as well
    ids, probs, status = run(batch, None, history, penalty)
    assert list(ids[1:5]) == [-1] * 4 and np.all(np.isnan(probs[1:5]))
    want = prepass.sample_processed(batch.values, batch.params, 5, 2, history=history, penalty=penalty)
    compare_sampler(want, ids, probs).check()
    assert status & binding.ROW_BAD_PARAMS


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_prepass_equals_smp_sample(dtype):
    # with no mask and no penalty the pre-pass path gives smp_sample's ids and
    # probabilities exactly (both are exact; one streams, one reads rows again)
    batch = workloads.random_sampler_batch(40, 20011, dtype=dtype, seed=8, kinds="mixed")
    logits = device_logits(batch.data, dtype)
    a = binding.sample(logits, batch.params, 9, 4)
    b = binding.sample_processed(logits, batch.params, 9, 4)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1], b[1]) or torch.allclose(a[1], b[1], rtol=1e-6, equal_nan=True)
    assert int(a[2].cpu()[0]) == int(b[2].cpu()[0])


VOCAB = ["[", "]", ","] + [str(d) for d in range(10)] + ["a"]


def grammar_words(prefix):
    if not prefix:
        ok = [t == "[" for t in VOCAB]
    elif prefix[-1] in {"[", ","}:
        ok = [t.isdigit() for t in VOCAB]
    elif prefix[-1].isdigit():
        ok = [t in {"]", ","} for t in VOCAB]
    else:
        ok = [False] * len(VOCAB)
    w = 0
    for i, a in enumerate(ok):
        w |= int(a) << i
    return np.array([w], dtype=np.uint32), np.array(ok)


def test_tiny_grammar_generation():
    # Listing 39.3's grammar '[' digit (',' digit)* ']' drives the mask step by
    # step; every sampled string is in the language
    rows = 64
    rng = np.random.default_rng(11)
    prefixes = [""] * rows
    for step in range(12):
        z = rng.normal(0, 2, (rows, len(VOCAB))).astype(np.float32)
        words = np.stack([grammar_words(p)[0] for p in prefixes])
        logits = torch.from_numpy(z).cuda()
        prm = workloads.make_params(rows, temperature=1.0)
        ids, _, _ = binding.sample_processed(logits, prm, 1, step,
                                             torch.from_numpy(words.view(np.int32)).cuda())
        ids = ids.cpu().numpy()
        for r in range(rows):
            ok = grammar_words(prefixes[r])[1]
            if not ok.any():
                assert ids[r] == -1
                continue
            assert ok[ids[r]]
            prefixes[r] += VOCAB[ids[r]]
    for p in prefixes:
        assert p.startswith("[")
        body = p[1:].rstrip("]")
        assert all(c.isdigit() or c == "," for c in body)
        assert ",," not in p and "[," not in p


def test_large_vocab_with_penalty_sampled_rows():
    # the headline batch (B 256, V 128256 bf16, mixed knobs) with a penalty
    # and a mask, checked on a sample of rows the oracle recomputes
    batch = workloads.sampler_workload("large_vocab")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=1, mask_density=(0.8, 1.0))
    ids, probs, status = run(batch, allowed, history, penalty, seed=0, offset=0)
    rows = list(range(0, 256, 9)) + [255]
    want = prepass.sample_processed(batch.values, batch.params, 0, 0, dtype="bf16", allowed=allowed,
                                    history=history, penalty=penalty, rows=rows)
    compare_sampler(want, ids, probs).check()


# ------------------------------------------------------------------ in place (smp_logit_prepass)


def storage_bits(values, dtype):
    v = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32)
    return (v >> 16).astype(np.uint16) if dtype == "bf16" else v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [31, 1000, 32000, 50021])
def test_inplace_prepass_is_bit_exact(dtype, vocab):
    batch = workloads.random_sampler_batch(12, vocab, dtype=dtype, seed=vocab % 31, kinds="mixed")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=vocab % 7)
    penalty[3] = 0.0                      # invalid: the row becomes NaN
    logits = device_logits(batch.data, dtype)
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
    status = binding.logit_prepass(logits, to(allowed, np.int32), to(history, np.int32), to(penalty, np.float32))
    torch.cuda.synchronize()
    assert int(status.cpu()[0]) == binding.ROW_BAD_PARAMS
    got = logits.cpu().view(torch.int16 if dtype == "bf16" else torch.int32).numpy()
    got = got.view(np.uint16 if dtype == "bf16" else np.uint32)
    for b in range(12):
        if b == 3:
            vals = got[b].astype(np.uint32) << 16 if dtype == "bf16" else got[b]
            assert np.all(np.isnan(vals.view(np.float32)))
            continue
        want = prepass.prepare_row(batch.values[b], dtype, allowed[b], history[b], penalty[b])
        assert np.array_equal(got[b], storage_bits(want, dtype)), b


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_inplace_prepass_then_sample(dtype):
    batch = workloads.random_sampler_batch(32, 20011, dtype=dtype, seed=21, kinds="mixed")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=22)
    logits = device_logits(batch.data, dtype)
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
    binding.logit_prepass(logits, to(allowed, np.int32), to(history, np.int32), to(penalty, np.float32))
    ids, probs, status = binding.sample(logits, batch.params, 6, 1)
    torch.cuda.synchronize()
    want = prepass.sample_processed(batch.values, batch.params, 6, 1, dtype=dtype, allowed=allowed,
                                    history=history, penalty=penalty)
    compare_sampler(want, ids.cpu().numpy(), probs.cpu().numpy()).check()
    # the row with no allowed token has no finite logit
    assert int(status.cpu()[0]) == binding.ROW_NONFINITE
    # and the out-of-place call gives the same ids
    fresh = device_logits(batch.data, dtype)
    ids2, _, _ = binding.sample_processed(fresh, batch.params, 6, 1, to(allowed, np.int32),
                                          to(history, np.int32), to(penalty, np.float32))
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2)


def test_more_rows_than_resident_ctas_with_prepass():
    # more rows than CTAs that fit on the GPU: each CTA takes several rows,
    # and its copies run ahead into the next row while the pre-pass state is
    # rebuilt per row
    batch = workloads.random_sampler_batch(700, 3001, dtype="bf16", seed=91, kinds="mixed")
    allowed, history, penalty = workloads.prepass_inputs(batch.values, seed=92)
    ids, probs, status = run(batch, allowed, history, penalty)
    rows = list(range(0, 700, 7)) + [699]
    want = prepass.sample_processed(batch.values, batch.params, 5, 2, dtype="bf16", allowed=allowed,
                                    history=history, penalty=penalty, rows=rows)
    compare_sampler(want, ids, probs).check()
