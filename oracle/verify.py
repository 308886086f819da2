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

Variants:

* temperature T > 0 on both distributions, p_T = softmax(z_p / T) and
  q_T = softmax(z_q / T), with the accept rule unchanged -- "Speculative
  decoding -- Hinglish notes", section "Temperature and Sampling";
* greedy verification (T = 0 or the greedy flag): a draft is kept when it is
  the target's top token (lowest id on ties), so the output is the target's
  own greedy decoding; at the first mismatch the target's top token is
  emitted, and if all K are kept the top token of position K -- "Inference:
  Sampling, the KV Cache, Speculative Decoding and int8", section
  "Speculative decoding";
* filters (top-k, top-p, min-p with the sampler's rules) on both
  distributions: p and q become the renormalised filtered distributions of
  eq. 39.2 at temperature T, computed exactly as the sampler computes them,
  and the accept, residual and bonus rules run on those.  The same section
  "Temperature and Sampling" says only that top-k and nucleus sampling act on
  the adjusted distribution around acceptance sampling; the reading taken is
  that both p and q are filtered, so that the output follows the target's
  filtered distribution, as the exactness argument of eq. 39.4 requires.

Readings taken where the pages leave a step open: by default temperature 1
and no filters on p and q; the
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
from .sampler import (ROW_BAD_PARAMS, ROW_NONFINITE, ROW_OK, filtered_distribution, is_greedy, logits_to_f64,
                      row_params_valid, walk)

Q_FLOOR = 1e-300


def softmax64(row, temperature=1.0):
    """Stable softmax of one logit row divided by the temperature, in float64."""
    z = logits_to_f64(row) / float(temperature)
    w = np.exp(z - np.max(z))
    return w / np.sum(w)


def top_token(row):
    """The arg-max of one logit row, lowest id on ties (NaN counts as -inf)."""
    z = logits_to_f64(row)
    return int(np.flatnonzero(z == np.max(z))[0])


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


def _distribution(row, temperature, filters):
    """p (or q) of one position: softmax(z / T), or, with filters, the
    renormalised filtered distribution of eq. 39.2 computed as the sampler
    does; returns (distribution, smallest filter margin)."""
    if filters is None:
        return softmax64(row, temperature), math.inf
    top_k, top_p, min_p = filters
    _, _, p_tilde, diag = filtered_distribution(row, temperature, top_k, top_p, min_p)
    return p_tilde, min(diag["topp_margin"], diag["minp_margin"])


def acceptance_rates(p_rows, q_rows, temperature=1.0, filters=None):
    """alpha_i = sum_x min(p_i(x), q_i(x)) for every draft position i: the
    probability that position i's proposal is kept ("Decoding & Speculative
    Sampling", section 39.4 and Listing 39.5), on the distributions the
    verifier compares (temperature and filters applied)."""
    out = []
    for i in range(len(q_rows)):
        p, _ = _distribution(p_rows[i], temperature, filters)
        q, _ = _distribution(q_rows[i], temperature, filters)
        out.append(float(np.sum(np.minimum(p, q))))
    return out


def verify_row(p_rows, q_rows, drafts, uniforms, temperature=1.0, greedy=False, filters=None):
    """Verify one batch row.

    p_rows:   [K+1, V] target logits; q_rows: [K, V] draft logits;
    drafts:   K draft token ids; uniforms: K+1 values (accept tests, then the
              final draw; unused when greedy);
    temperature, greedy: the variants above (temperature 0 means greedy);
    filters:  None, or (top_k, top_p, min_p) applied to every p and q row.
    Returns a dict with accepted (int), ids (list of K+1 ints, -1 past the
    emitted tokens), status, and the margins accept_margin (smallest |u_i -
    p/q| over the accept tests made), draw_margin and filter_margin (the
    smallest top-p or min-p margin of the distributions used).
    """
    k = len(drafts)
    vocab = p_rows.shape[1]
    out = {"accepted": -1, "ids": [-1] * (k + 1), "status": ROW_OK,
           "accept_margin": math.inf, "draw_margin": math.inf, "filter_margin": math.inf}
    greedy = bool(greedy) or float(temperature) == 0.0
    # greedy verification reads no draft distribution, so only p is checked
    for row in list(p_rows) + ([] if greedy else list(q_rows)):
        if not math.isfinite(np.max(logits_to_f64(row))):
            out["status"] = ROW_NONFINITE
            return out
    if any(not (0 <= int(x) < vocab) for x in drafts):
        out["status"] = ROW_BAD_PARAMS
        return out
    emitted = []
    if greedy:
        for i in range(k + 1):
            top = top_token(p_rows[i])
            if i < k and int(drafts[i]) == top:
                emitted.append(top)
                continue
            out["accepted"] = i
            out["ids"] = emitted + [top] + [-1] * (k - i)
            return out
    for i in range(k):
        p, mp = _distribution(p_rows[i], temperature, filters)
        q, mq = _distribution(q_rows[i], temperature, filters)
        out["filter_margin"] = min(out["filter_margin"], mp, mq)
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
    p_bonus, mb = _distribution(p_rows[k], temperature, filters)
    out["filter_margin"] = min(out["filter_margin"], mb)
    token = walk(p_bonus, uniforms[k])
    out["draw_margin"] = _draw_margin(p_bonus, uniforms[k])
    out["accepted"] = k
    out["ids"] = emitted + [token]
    return out


def _draw_margin(dist, u):
    running = np.cumsum(dist)[dist > 0]
    return float(np.min(np.abs(np.concatenate(([0.0], running)) - u)))


def row_mode(prm, vocab):
    """Status, temperature, greedy flag and filters of one batch row's knobs.

    prm: a record with fields temperature, top_k, top_p, min_p, greedy (the
    sampler's knobs, with the sampler's validity rules).  Greedy (the flag, or
    T = 0) ignores the other knobs, as in sampling.  Otherwise the filters
    that are on (0 < top_k < V, top_p < 1, 0 < min_p < 1) apply to every p
    and q row, or filters is None when all are off.
    """
    t, g = float(prm["temperature"]), int(prm["greedy"])
    if is_greedy(t, g):
        return ROW_OK, 0.0, True, None
    if not row_params_valid(t, prm["top_k"], prm["top_p"], prm["min_p"]):
        return ROW_BAD_PARAMS, t, False, None
    k, top_p, min_p = int(prm["top_k"]), float(prm["top_p"]), float(prm["min_p"])
    if 0 < k < vocab or top_p < 1.0 or 0.0 < min_p < 1.0:
        return ROW_OK, t, False, (k, top_p, min_p)
    return ROW_OK, t, False, None


def spec_verify(p_logits, q_logits, draft_ids, seed, offset, rows=None, temperature=1.0, greedy=False,
                params=None, alpha=False, row_base=0):
    """Run verify_row over a batch (temperature and greedy for all its rows,
    or per row from `params`, one record per batch row, see row_mode).
    alpha: also return each row's acceptance rates ("alpha", K values; NaN
    for greedy and error rows, which compare no distributions).

    p_logits: [B, K+1, V]; q_logits: [B, K, V]; draft_ids: [B, K].
    Uniform for batch row b, draw d: philox.uniform(seed, offset, row_base + b, d)
    (row_base: global index of row 0 when the batch is one part of a larger one).
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
        us = [philox.uniform(seed, offset, int(row_base) + int(b), d) for d in range(k + 1)]
        if params is not None:
            status, t_row, g_row, f_row = row_mode(params[b], p_logits.shape[-1])
            if status != ROW_OK:
                res = {"accepted": -1, "ids": [-1] * (k + 1), "status": status, "accept_margin": math.inf,
                       "draw_margin": math.inf, "filter_margin": math.inf, "row": int(b)}
                if alpha:
                    res["alpha"] = [math.nan] * k
                results.append(res)
                continue
        else:
            t_row, g_row, f_row = temperature, greedy, None
        res = verify_row(p_logits[b], q_logits[b], draft_ids[b], us, t_row, g_row, f_row)
        if alpha:
            g_eff = bool(g_row) or float(t_row) == 0.0
            if res["status"] != ROW_OK or g_eff:
                res["alpha"] = [math.nan] * k
            else:
                res["alpha"] = acceptance_rates(p_logits[b], q_logits[b], t_row, f_row)
        res["row"] = int(b)
        results.append(res)
    return results
