"""fp64 oracle of the speculative-decoding verifier (test infrastructure).

Follows the accept / resample / bonus rule as the pages state it:

* each draft token x at position i is kept with probability
  min(1, p_i(x) / q_i(x)) -- "Decoding & Speculative Sampling", eq. 39.3, and
  "Efficient Inference & Compression", section "Speculative decoding", step 1;
  the test is u_i < p_i(x) / max(q_i(x), 1e-300), the floor on q that the
  one-token listing of section 39.4 uses;
* at the first rejection the later drafts are discarded and a replacement is
  drawn from r = max(0, p_i - q_i) / sum_y max(0, p_i(y) - q_i(y)) -- eq. 39.4,
  and "Speculative decoding -- Hinglish notes", section "The Algorithm
  (Step-by-Step)", step 3;
* if all K drafts are kept, one bonus token is drawn from the target's
  position-K distribution -- same step 3, and "Inference: Sampling, the KV
  Cache, Speculative Decoding and int8", section "Speculative decoding";
* every row of the batch accepts 0..K tokens on its own -- "Speculative
  decoding -- Hinglish notes", section "Batching Speculation".

Readings (listed in the design doc): temperature 1 and no filters on p and q; the
uniforms are Philox draws 0..K-1 for the K accept tests and draw K for the one
resample or bonus draw; if the residual has zero total mass (possible only
through rounding) the replacement is drawn from p_i; the walk is the sampler's
id-order inverse CDF; a row with a non-finite maximum in any of its 2K+1
logit rows, or a draft id outside [0, V), is an error row (accepted length -1,
all ids -1).

Test infrastructure only: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline leg may import it.
"""

import math

import numpy as np

from . import philox
from .sampler import ROW_BAD_PARAMS, ROW_NONFINITE, ROW_OK, logits_to_f64, walk

Q_FLOOR = 1e-300


def softmax64(row):
    """Stable softmax of one logit row in float64 (temperature 1)."""
    z = logits_to_f64(row)
    w = np.exp(z - np.max(z))
    return w / np.sum(w)


def accept_draft(p, q, x, u):
    """The accept test of eq. 39.3 for draft token x with uniform u."""
    return u < p[x] / max(q[x], Q_FLOOR)


def residual_distribution(p, q):
    """max(0, p - q) renormalised (eq. 39.4); p itself if the mass is zero."""
    r = np.maximum(p - q, 0.0)
    total = np.sum(r)
    if total > 0.0:
        return r / total
    return p


def verify_row(p_rows, q_rows, drafts, uniforms):
    """Verify one batch row.

    p_rows:   [K+1, V] target logits; q_rows: [K, V] draft logits;
    drafts:   K draft token ids; uniforms: K+1 values (accept tests, then the
              final draw).
    Returns a dict with accepted (int), ids (list of K+1 ints, -1 past the
    emitted tokens), status, and the margins accept_margin (smallest |u_i -
    p/q| over the accept tests made) and draw_margin.
    """
    k = len(drafts)
    vocab = p_rows.shape[1]
    out = {"accepted": -1, "ids": [-1] * (k + 1), "status": ROW_OK,
           "accept_margin": math.inf, "draw_margin": math.inf}
    for row in list(p_rows) + list(q_rows):
        if not math.isfinite(np.max(logits_to_f64(row))):
            out["status"] = ROW_NONFINITE
            return out
    if any(not (0 <= int(x) < vocab) for x in drafts):
        out["status"] = ROW_BAD_PARAMS
        return out
    emitted = []
    for i in range(k):
        p = softmax64(p_rows[i])
        q = softmax64(q_rows[i])
        x = int(drafts[i])
        ratio = p[x] / max(q[x], Q_FLOOR)
        out["accept_margin"] = min(out["accept_margin"], abs(uniforms[i] - ratio))
        if accept_draft(p, q, x, uniforms[i]):
            emitted.append(x)
            continue
        dist = residual_distribution(p, q)
        token = walk(dist, uniforms[k])
        out["draw_margin"] = _draw_margin(dist, uniforms[k])
        out["accepted"] = i
        out["ids"] = emitted + [token] + [-1] * (k - i)
        return out
    p_bonus = softmax64(p_rows[k])
    token = walk(p_bonus, uniforms[k])
    out["draw_margin"] = _draw_margin(p_bonus, uniforms[k])
    out["accepted"] = k
    out["ids"] = emitted + [token]
    return out


def _draw_margin(dist, u):
    running = np.cumsum(dist)[dist > 0]
    return float(np.min(np.abs(np.concatenate(([0.0], running)) - u)))


def spec_verify(p_logits, q_logits, draft_ids, seed, offset, rows=None):
    """Run verify_row over a batch.

    p_logits: [B, K+1, V]; q_logits: [B, K, V]; draft_ids: [B, K].
    Uniform for batch row b, draw d: philox.uniform(seed, offset, b, d).
    Returns a list of per-row dicts (with "row") in the order of `rows`.
    """
    p_logits = np.asarray(p_logits)
    q_logits = np.asarray(q_logits)
    draft_ids = np.asarray(draft_ids)
    k = draft_ids.shape[1]
    if rows is None:
        rows = range(p_logits.shape[0])
    results = []
    for b in rows:
        us = [philox.uniform(seed, offset, int(b), d) for d in range(k + 1)]
        res = verify_row(p_logits[b], q_logits[b], draft_ids[b], us)
        res["row"] = int(b)
        results.append(res)
    return results
