"""Oracle of the logit pre-pass before sampling (test infrastructure).

Two transforms of a row's logits, applied before temperature, filters and the
draw of oracle.sampler:

* repetition penalty -- "Choosing the next word", section "The repetition
  penalty" (the CTRL rule): for each token i found among the last tokens of
  the text, z_i <- z_i / r if z_i > 0, else z_i * r;
* constraint mask -- "Decoding & Speculative Sampling", section 39.3 and
  Listing 39.3: every token outside the allowed set gets the logit -inf, so
  the softmax is the model's distribution conditioned on the allowed set.

Readings taken where the pages leave a step open:

* order: the penalty acts on the raw logits (the sign test is on the raw
  value), then the mask, then temperature and the filters as in sampling;
* each distinct token id of the history is penalised once (duplicates in the
  window change nothing); history entries outside [0, V) are padding;
* the penalised value is computed in binary32 (one correctly rounded division
  or product) and stored in the logits' own precision (bf16 logits: rounded
  to the nearest bf16, ties to even), so that both sides order the same
  values;
* r must be finite and > 0 (r = 1 leaves the row unchanged); otherwise the
  row is an error row (bad knobs), greedy or not;
* the mask is a bit array per row, bit (i mod 32) of word i // 32 set when
  token i is allowed; an empty allowed set leaves no finite logit, which is
  the sampler's error row for a non-finite maximum (the pages call an empty
  allowed set an invalid decoder state).

Test infrastructure only: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline leg may import it.
"""

import math

import numpy as np

from . import philox
from .sampler import ROW_BAD_PARAMS, sample_row


def round_to_bf16(x):
    """Nearest bf16 value of a binary32 number (ties to even), as float32.

    bf16 keeps the upper 16 bits of binary32: add half of the dropped part's
    range (0x7FFF plus the lowest kept bit, for ties to even) and truncate.
    NaN stays NaN; infinities stay infinite.
    """
    x = np.float32(x)
    if math.isnan(float(x)):
        return np.float32(np.nan)
    bits = int(np.array(x, dtype=np.float32).view(np.uint32))
    lsb = (bits >> 16) & 1
    bits = ((bits + 0x7FFF + lsb) >> 16) << 16
    return np.array(bits & 0xFFFFFFFF, dtype=np.uint32).view(np.float32)[()]


def penalize(z, r, dtype="f32"):
    """The repetition penalty of one logit: z / r for z > 0, z * r otherwise."""
    z = np.float32(z)
    r = np.float32(r)
    with np.errstate(invalid="ignore", over="ignore"):
        out = np.float32(z / r) if z > 0 else np.float32(z * r)
    return round_to_bf16(out) if dtype == "bf16" else out


def allowed_mask(words, vocab):
    """Boolean [vocab] allowed set from one row of 32-bit mask words."""
    words = np.asarray(words, dtype=np.uint32)
    ids = np.arange(vocab)
    return ((words[ids // 32] >> (ids % 32).astype(np.uint32)) & 1).astype(bool)


def penalty_valid(r):
    r = float(r)
    return math.isfinite(r) and r > 0.0


def prepare_row(row, dtype="f32", allowed_words=None, history=None, penalty=1.0):
    """The logits the sampler sees for one row (float32 array)."""
    z = np.array(row, dtype=np.float32).copy()
    vocab = z.size
    if history is not None and float(penalty) != 1.0:
        for i in sorted({int(h) for h in history if 0 <= int(h) < vocab}):
            z[i] = penalize(z[i], penalty, dtype)
    if allowed_words is not None:
        z[~allowed_mask(allowed_words, vocab)] = -np.inf
    return z


def sample_processed(logits, params, seed, offset, dtype="f32", allowed=None, history=None, penalty=None,
                     rows=None, row_base=0):
    """oracle.sampler.sample on pre-processed rows.

    allowed: [B, ceil(V / 32)] uint32 or None; history: [B, H] int or None;
    penalty: [B] float or None (no penalty); row_base: global index of row 0
    (the uniform of row b is drawn at counter row row_base + b).  Returns
    per-row result dicts.
    """
    logits = np.asarray(logits)
    if rows is None:
        rows = range(logits.shape[0])
    results = []
    for b in rows:
        prm = params[b]
        u = philox.uniform(seed, offset, int(row_base) + int(b), 0)
        r = 1.0 if penalty is None else float(penalty[b])
        if not penalty_valid(r):
            res = {"token": -1, "prob": math.nan, "status": ROW_BAD_PARAMS, "kept": 0,
                   "topp_margin": math.inf, "minp_margin": math.inf, "draw_margin": math.inf}
        else:
            z = prepare_row(logits[b], dtype, None if allowed is None else allowed[b],
                            None if history is None else history[b], r)
            res = sample_row(z, prm["temperature"], prm["top_k"], prm["top_p"], prm["min_p"],
                             prm["greedy"], u)
        res["row"] = int(b)
        res["u"] = u
        results.append(res)
    return results
