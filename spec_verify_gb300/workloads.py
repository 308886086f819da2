"""Seeded synthetic workloads for the sampler and the verifier.

This module only makes inputs: logits, per-row knobs and their memory layout.
It holds none of the method's arithmetic (no softmax, masking or drawing), so
the CUDA path's tests and bench and the oracle can both consume it.

Workload recipes (each seeded with numpy.random.default_rng):

* "basic":      B=4, V=8192, fp32 logits i.i.d. N(0, 2^2); every row T=0.8,
                top_k=50, top_p=0.9, min_p=0.05.
* "mixed":      B=64, V=32000, bf16 Zipf-headed logits (below); per-row knobs
                T ~ U[0.7, 1.0], top_k in {0, 40, 100}, top_p in {1.0, 0.9,
                0.95}, min_p in {0, 0.05, 0.1}; rows with b % 8 == 7 greedy.
* "large_vocab": B=256, V=128256, bf16 Zipf-headed logits; rows b % 4 in {0, 1}
                min_p=0.1 at T=1, b % 4 == 2 greedy, b % 4 == 3 T=0.7 with
                top_k=40.
* "verify":     B=32, K=4, V=32000, fp32; G ~ N(0, 2^2) of shape [B, K+1, V];
                draft logits q = G[:, :K], target logits p = G + N(0, 1^2).
                Draft ids are drawn from q by the caller (T=1, no filters,
                seed 1, offset 0).
* "flat_nucleus": B=1024, V=152064, bf16 i.i.d. N(0, 0.3^2); T=1, top_p=0.95.

Zipf-headed logits: for each row, rank r = 1..V gets log(r^-1.1); a seeded
random permutation per row assigns ranks to token ids; N(0, 0.5^2) noise is
added and the result is rounded to bf16 (round to nearest even).

Logit seeds are 1000 + id and knob seeds 2000 + id, id = 1..5 in the order
above.
"""

import numpy as np

# Matches the C struct smp_row_params (20 bytes, little endian).
PARAMS_DTYPE = np.dtype([("temperature", "<f4"), ("top_k", "<i4"),
                         ("top_p", "<f4"), ("min_p", "<f4"), ("greedy", "<i4")])

WORKLOADS = ("basic", "mixed", "large_vocab", "verify", "flat_nucleus")
WORKLOAD_ID = {name: i + 1 for i, name in enumerate(WORKLOADS)}


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    rounded = (u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = ((u[nan] >> 16) | 0x0040).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_params(batch, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0, greedy=0):
    """A params array with every row set to the same knobs."""
    prm = np.zeros(batch, dtype=PARAMS_DTYPE)
    prm["temperature"] = temperature
    prm["top_k"] = top_k
    prm["top_p"] = top_p
    prm["min_p"] = min_p
    prm["greedy"] = greedy
    return prm


def zipf_logits_f32(rng, batch, vocab, s=1.1, noise=0.5):
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    head = (-s * np.log(ranks)).astype(np.float64)
    out = np.empty((batch, vocab), dtype=np.float32)
    for b in range(batch):
        perm = rng.permutation(vocab)
        row = np.empty(vocab, dtype=np.float64)
        row[perm] = head
        row += rng.normal(0.0, noise, size=vocab)
        out[b] = row.astype(np.float32)
    return out


class Batch:
    """A sampler batch: logits as stored on the device plus widened float32.

    dtype: "f32" or "bf16"; data: array of the device layout (float32 or the
    uint16 bf16 bit patterns), shape [B, V]; values: float32 copy of the logits
    (exact); params: PARAMS_DTYPE array [B]; seed/offset: Philox key and step.
    """

    def __init__(self, name, dtype, data, params, seed=0, offset=0):
        self.name = name
        self.dtype = dtype
        self.data = data
        self.params = params
        self.seed = seed
        self.offset = offset

    @property
    def shape(self):
        return self.data.shape

    @property
    def values(self):
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.data)
        return self.data


def sampler_workload(name, batch=None):
    """Build one of the sampler workloads ("basic", "mixed", "large_vocab",
    "flat_nucleus").  `batch` truncates the batch to its first rows."""
    wid = WORKLOAD_ID[name]
    rng = np.random.default_rng(1000 + wid)
    prng = np.random.default_rng(2000 + wid)
    if name == "basic":
        B, V = 4, 8192
        logits = rng.normal(0.0, 2.0, size=(B, V)).astype(np.float32)
        params = make_params(B, temperature=0.8, top_k=50, top_p=0.9, min_p=0.05)
        out = Batch(name, "f32", logits, params)
    elif name == "mixed":
        B, V = 64, 32000
        data = f32_to_bf16_bits(zipf_logits_f32(rng, B, V))
        params = make_params(B)
        params["temperature"] = prng.uniform(0.7, 1.0, size=B).astype(np.float32)
        params["top_k"] = prng.choice([0, 40, 100], size=B)
        params["top_p"] = prng.choice(np.array([1.0, 0.9, 0.95], dtype=np.float32), size=B)
        params["min_p"] = prng.choice(np.array([0.0, 0.05, 0.1], dtype=np.float32), size=B)
        params["greedy"] = (np.arange(B) % 8 == 7).astype(np.int32)
        out = Batch(name, "bf16", data, params)
    elif name == "large_vocab":
        B, V = 256, 128256
        data = f32_to_bf16_bits(zipf_logits_f32(rng, B, V))
        params = make_params(B)
        kind = np.arange(B) % 4
        params["min_p"][kind < 2] = 0.1
        params["greedy"][kind == 2] = 1
        params["temperature"][kind == 3] = 0.7
        params["top_k"][kind == 3] = 40
        out = Batch(name, "bf16", data, params)
    elif name == "flat_nucleus":
        B, V = 1024, 152064
        data = f32_to_bf16_bits(rng.normal(0.0, 0.3, size=(B, V)).astype(np.float32))
        params = make_params(B, temperature=1.0, top_p=0.95)
        out = Batch(name, "bf16", data, params)
    else:
        raise ValueError(f"unknown sampler workload {name!r}")
    if batch is not None:
        out.data = out.data[:batch].copy()
        out.params = out.params[:batch].copy()
    return out


class VerifyBatch:
    """Verifier inputs: p [B, K+1, V], q [B, K, V] (device layout), seeds."""

    def __init__(self, name, dtype, p, q, seed=0, offset=0, draft_seed=1, draft_offset=0):
        self.name = name
        self.dtype = dtype
        self.p = p
        self.q = q
        self.seed = seed
        self.offset = offset
        self.draft_seed = draft_seed
        self.draft_offset = draft_offset

    @property
    def shape(self):
        B, K1, V = self.p.shape
        return B, K1 - 1, V

    def values(self, which):
        arr = self.p if which == "p" else self.q
        if self.dtype == "bf16":
            return bf16_bits_to_f32(arr)
        return arr


def verify_workload(batch=32, k=4, vocab=32000, dtype="f32", seed_id=None):
    """The "verify" workload: G ~ N(0, 2^2), q = G[:, :K], p = G + N(0, 1^2)."""
    wid = WORKLOAD_ID["verify"] if seed_id is None else seed_id
    rng = np.random.default_rng(1000 + wid)
    g = rng.normal(0.0, 2.0, size=(batch, k + 1, vocab)).astype(np.float32)
    p = (g + rng.normal(0.0, 1.0, size=g.shape)).astype(np.float32)
    q = np.ascontiguousarray(g[:, :k])
    if dtype == "bf16":
        p, q = f32_to_bf16_bits(p), f32_to_bf16_bits(q)
    return VerifyBatch("verify", dtype, p, q)


def random_sampler_batch(batch, vocab, dtype="bf16", seed=0, kinds="mixed"):
    """Small seeded batches for parity tests: Zipf-headed logits and knob mixes.

    kinds: "mixed" draws every knob at random per row (including greedy and
    off values); or one of "greedy", "minp", "topk", "topp", "plain".
    """
    rng = np.random.default_rng(50_000 + seed)
    logits = zipf_logits_f32(rng, batch, vocab)
    prm = make_params(batch)
    if kinds == "mixed":
        prm["temperature"] = rng.uniform(0.5, 1.5, size=batch)
        prm["top_k"] = rng.choice([0, 1, 5, 40, 300, vocab], size=batch)
        prm["top_p"] = rng.choice(np.array([1.0, 0.5, 0.9, 0.95, 0.99], dtype=np.float32), size=batch)
        prm["min_p"] = rng.choice(np.array([0.0, 0.01, 0.05, 0.2], dtype=np.float32), size=batch)
        prm["greedy"] = (rng.uniform(size=batch) < 0.1).astype(np.int32)
    elif kinds == "greedy":
        prm["greedy"] = 1
    elif kinds == "minp":
        prm["min_p"] = rng.choice(np.array([0.02, 0.1, 0.5], dtype=np.float32), size=batch)
        prm["temperature"] = rng.uniform(0.5, 1.5, size=batch)
    elif kinds == "topk":
        prm["top_k"] = rng.choice([1, 2, 40, 100, 1000], size=batch)
        prm["temperature"] = rng.uniform(0.5, 1.5, size=batch)
    elif kinds == "topp":
        prm["top_p"] = rng.choice(np.array([0.3, 0.9, 0.95, 0.999], dtype=np.float32), size=batch)
        prm["temperature"] = rng.uniform(0.5, 1.5, size=batch)
    elif kinds == "plain":
        prm["temperature"] = rng.uniform(0.5, 1.5, size=batch)
    else:
        raise ValueError(kinds)
    if dtype == "bf16":
        return Batch(f"random-{kinds}", "bf16", f32_to_bf16_bits(logits), prm)
    return Batch(f"random-{kinds}", "f32", logits, prm)


def prepass_inputs(values, seed=0, history_len=64, mask_density=(0.3, 0.95)):
    """Seeded inputs of the logit pre-pass for a [B, V] batch of logit values.

    Returns (allowed [B, ceil(V/32)] uint32, history [B, H] int32, penalty [B]
    float32).  Row densities of allowed tokens are drawn from mask_density;
    row 0 allows one token only, and the last row of batches of 8 or more
    allows none.  Histories hold some of the row's 32 highest-logit ids (so
    that the penalty changes the outcome), random ids, repeats, and padding
    (-1 and ids past V).  Penalties come from {1.0, 1.1, 1.3, 2.0, 0.8}.
    """
    values = np.asarray(values, dtype=np.float32)
    batch, vocab = values.shape
    rng = np.random.default_rng(70_000 + seed)
    words = (vocab + 31) // 32
    allowed = np.zeros((batch, words), dtype=np.uint32)
    for b in range(batch):
        dens = rng.uniform(*mask_density)
        keep = rng.uniform(size=vocab) < dens
        if b == 0:
            keep[:] = False
            keep[rng.integers(vocab)] = True
        if batch >= 8 and b == batch - 1:
            keep[:] = False
        ids = np.flatnonzero(keep)
        np.bitwise_or.at(allowed[b], ids // 32, (np.uint32(1) << (ids % 32).astype(np.uint32)))
    history = np.full((batch, history_len), -1, dtype=np.int32)
    for b in range(batch):
        top = np.argsort(-values[b], kind="stable")[:32]
        picks = list(rng.choice(top, size=min(12, top.size), replace=False))
        picks += list(rng.integers(0, vocab, size=history_len // 2))
        picks += picks[:4]                      # repeats
        picks += [vocab + 3, -5]                # padding past either end
        rng.shuffle(picks)
        n = min(history_len, len(picks))
        history[b, :n] = np.array(picks[:n], dtype=np.int64).astype(np.int32)
    penalty = rng.choice(np.array([1.0, 1.1, 1.3, 2.0, 0.8], dtype=np.float32), size=batch)
    return allowed, history, penalty
