"""fp64 oracle of the batched next-token sampler (test infrastructure).

Plain, slow and written to be checked against the pages by eye.  Every step
follows one passage:

* temperature divides the logits before the softmax -- "Decoding & Speculative
  Sampling", section 39.2 (and "Choosing the next word", section "Temperature:
  one dial for boldness");
* the softmax subtracts the row maximum before exponentiating -- section 39.2,
  Listing 39.2 (stable softmax);
* top-k keeps the k most likely tokens, top-p keeps the shortest most-likely
  prefix whose cumulative probability reaches p, min-p keeps tokens with
  p_i >= min_p * max_j p_j -- section 39.2 and "Inference: Sampling, the KV
  Cache, Speculative Decoding and int8", section "Picking the next token";
* the kept set S is renormalised, p~_i = p_i 1{i in S} / sum_j p_j 1{j in S}
  -- eq. 39.2;
* greedy is the arg-max, the T -> 0 limit -- section 39.1 and 39.2;
* a token is drawn by walking the kept tokens, adding their probabilities, and
  stopping at the first one whose running total passes u -- "Choosing the next
  word", section "Where the randomness comes from, and where it stops".

Readings taken where the pages leave a step open:

* all three masks are computed on the same post-temperature p and intersected
  (eq. 39.2, Listing 39.2); each mask is a prefix of the order
  (logit descending, token id ascending), so S is the shortest of them;
* ties are broken by the lower token id, and top-k keeps exactly k tokens;
* top-p keeps the shortest prefix with cumulative sum >= top_p, never fewer than
  one token; top_p >= 1 switches it off;
* min-p is active for 0 < min_p < 1, top-k for 0 < top_k < V;
* temperature 0 or the greedy flag gives the arg-max (lowest id on ties);
* NaN logits count as -inf; a row whose maximum is not finite (all -inf/NaN,
  or any +inf) is an error row: token -1;
* invalid knobs (T < 0, T non-finite, top_k < 0, top_p < 0 or NaN, min_p < 0 or
  NaN) on a sampling row give an error row;
* the walk runs in token-id order with a strict "passes" (>), so tokens of zero
  probability are never drawn; if rounding leaves u past the last running total
  the last kept token is taken.

This module is test infrastructure.  Only tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline leg may import it; nothing on the product path does.
"""

import math

import numpy as np

from . import philox

# Error outcomes for one row (also OR-ed into the CUDA path's status word).
ROW_OK = 0
ROW_BAD_PARAMS = 1
ROW_NONFINITE = 2


def logits_to_f64(row):
    """Logits as float64 with NaN replaced by -inf (exact for bf16 and fp32)."""
    z = np.asarray(row, dtype=np.float64).copy()
    z[np.isnan(z)] = -np.inf
    return z


def softmax_with_temperature(z, temperature):
    """p = softmax(z / T) in float64, subtracting the maximum first."""
    x = z / float(temperature)
    shifted = x - np.max(x)
    w = np.exp(shifted)
    return w / np.sum(w)


def descending_order(z):
    """Token ids sorted by logit descending, ties by ascending id."""
    ids = np.arange(z.size)
    # np.lexsort sorts by the last key first: primary -z (ascending), then id.
    return np.lexsort((ids, -z))


def keep_top_k(order, k):
    """Boolean mask of the first k tokens of `order`."""
    keep = np.zeros(order.size, dtype=bool)
    keep[order[:k]] = True
    return keep


def nucleus_length(p_sorted, top_p):
    """Length of the shortest prefix whose cumulative probability is >= top_p.

    The cumulative sum is taken left to right in float64.  At least one token
    is kept; if no prefix reaches top_p (rounding) the whole vocabulary is.
    """
    cum = np.cumsum(p_sorted)
    reached = np.flatnonzero(cum >= top_p)
    if reached.size == 0:
        return p_sorted.size
    return int(reached[0]) + 1


def keep_top_p(order, p, top_p):
    """Boolean mask of the nucleus: the first nucleus_length tokens of order."""
    length = nucleus_length(p[order], top_p)
    keep = np.zeros(order.size, dtype=bool)
    keep[order[:length]] = True
    return keep


def keep_min_p(p, min_p):
    """Boolean mask p_i >= min_p * max_j p_j."""
    return p >= float(min_p) * np.max(p)


def walk(weights, u):
    """Index drawn by the inverse-CDF walk in id order.

    `weights` are the (renormalised) probabilities, zero outside the kept set.
    Returns the first index whose running total is strictly greater than u; if
    rounding leaves u beyond the final total, the last index of positive weight.
    """
    running = np.cumsum(weights)
    past = np.flatnonzero(running > u)
    if past.size:
        return int(past[0])
    return int(np.flatnonzero(weights > 0)[-1])


def row_params_valid(temperature, top_k, top_p, min_p):
    """Validity of the knobs of a sampling (non-greedy) row."""
    t = float(temperature)
    if not (math.isfinite(t) and t > 0.0):
        return False
    if int(top_k) < 0:
        return False
    if math.isnan(float(top_p)) or float(top_p) < 0.0:
        return False
    if math.isnan(float(min_p)) or float(min_p) < 0.0:
        return False
    return True


def is_greedy(temperature, greedy):
    return int(greedy) != 0 or float(temperature) == 0.0


def filtered_distribution(row, temperature, top_k=0, top_p=1.0, min_p=0.0):
    """p (after temperature), the kept mask S and p~ of eq. 39.2 for one row.

    Returns (p, keep, p_tilde, diag) where diag holds the margins the parity
    tests use to excuse rows decided by rounding.
    """
    z = logits_to_f64(row)
    vocab = z.size
    p = softmax_with_temperature(z, temperature)
    order = descending_order(z)
    keep = np.ones(vocab, dtype=bool)
    diag = {"topp_margin": math.inf, "minp_margin": math.inf}
    if 0 < int(top_k) < vocab:
        keep &= keep_top_k(order, int(top_k))
    if float(top_p) < 1.0:
        keep &= keep_top_p(order, p, float(top_p))
        cum = np.cumsum(p[order])
        diag["topp_margin"] = float(np.min(np.abs(cum - float(top_p))))
    if 0.0 < float(min_p) < 1.0:
        keep &= keep_min_p(p, float(min_p))
        diag["minp_margin"] = float(np.min(np.abs(p / np.max(p) - float(min_p))))
    kept_mass = np.sum(np.where(keep, p, 0.0))
    p_tilde = np.where(keep, p, 0.0) / kept_mass
    return p, keep, p_tilde, diag


def sample_row(row, temperature, top_k, top_p, min_p, greedy, u):
    """Draw one token for one row.

    Returns a dict: token (int, -1 on an error row), prob (p~ of the token,
    1.0 for greedy), status (ROW_*), kept (|S|), and the margins topp_margin,
    minp_margin, draw_margin (distance from u to the nearest running total).
    """
    z = logits_to_f64(row)
    out = {"token": -1, "prob": math.nan, "status": ROW_OK, "kept": 0,
           "topp_margin": math.inf, "minp_margin": math.inf,
           "draw_margin": math.inf}
    zmax = np.max(z)
    if not math.isfinite(zmax):
        out["status"] = ROW_NONFINITE
        return out
    if is_greedy(temperature, greedy):
        out["token"] = int(np.flatnonzero(z == zmax)[0])
        out["prob"] = 1.0
        out["kept"] = 1
        return out
    if not row_params_valid(temperature, top_k, top_p, min_p):
        out["status"] = ROW_BAD_PARAMS
        return out
    _, keep, p_tilde, diag = filtered_distribution(z, temperature, top_k, top_p, min_p)
    token = walk(p_tilde, u)
    running = np.cumsum(p_tilde)[keep]
    boundaries = np.concatenate(([0.0], running))
    out.update(diag)
    out["token"] = token
    out["prob"] = float(p_tilde[token])
    out["kept"] = int(np.count_nonzero(keep))
    out["draw_margin"] = float(np.min(np.abs(boundaries - u)))
    return out


def sample(logits, params, seed, offset, rows=None, row_base=0):
    """Run sample_row over a [B, V] batch.

    logits: array [B, V] of float32 values (bf16 logits widened exactly).
    params: structured array with fields temperature, top_k, top_p, min_p,
            greedy (one record per row).
    rows:   optional subset of row indices (the Philox counter uses the row's
            own index, so any subset gives the same per-row results).
    row_base: global index of row 0 when the batch is one part of a larger
            batch: row b draws its uniform at counter row row_base + b, so a
            batch split into parts gives the tokens of the whole.
    Returns a list of per-row result dicts in the order of `rows`.
    """
    logits = np.asarray(logits)
    if rows is None:
        rows = range(logits.shape[0])
    results = []
    for b in rows:
        prm = params[b]
        u = philox.uniform(seed, offset, int(row_base) + int(b), 0)
        res = sample_row(logits[b], prm["temperature"], prm["top_k"],
                         prm["top_p"], prm["min_p"], prm["greedy"], u)
        res["row"] = int(b)
        res["u"] = u
        results.append(res)
    return results


def filtered_rows(logits, params, rows=None):
    """p~ (eq. 39.2) and |S| for each requested row, greedy rows as one-hot.

    Error rows give an all-NaN p~ and kept = 0.
    """
    logits = np.asarray(logits)
    if rows is None:
        rows = range(logits.shape[0])
    out = []
    for b in rows:
        prm = params[b]
        z = logits_to_f64(logits[b])
        zmax = np.max(z)
        if not math.isfinite(zmax):
            out.append((np.full(z.size, np.nan), 0))
            continue
        if is_greedy(prm["temperature"], prm["greedy"]):
            onehot = np.zeros(z.size)
            onehot[np.flatnonzero(z == zmax)[0]] = 1.0
            out.append((onehot, 1))
            continue
        if not row_params_valid(prm["temperature"], prm["top_k"], prm["top_p"], prm["min_p"]):
            out.append((np.full(z.size, np.nan), 0))
            continue
        _, keep, p_tilde, _ = filtered_distribution(
            z, prm["temperature"], prm["top_k"], prm["top_p"], prm["min_p"])
        out.append((p_tilde, int(np.count_nonzero(keep))))
    return out
