"""fp64 oracle of one beam-search step's candidate selection (test infrastructure).

"Decoding & Speculative Sampling", section 39.1, eq. 39.1 and Listing 39.1:
a prefix's score is the sum of its tokens' log-probabilities; every beam is
extended by every token, the candidate's score is the beam's score plus
log p(token | prefix), and the B highest-scoring candidates survive.
"Efficient Inference & Compression", section "Beam search", states the same
step (the k best of all extensions of the k beams).

Readings taken where the pages leave a step open:

* candidates are ordered by score, highest first; equal scores keep the order
  in which Listing 39.1 appends them (beam by beam, token by token), because
  its sort is stable: the lower flat index beam * V + token wins;
* log p is the log-softmax of the beam's logits at temperature 1 with no
  filters (the listing's softmax), computed as z - max z - log sum exp(z - max z);
* NaN logits count as -inf; a beam whose logits have no finite maximum, or a
  NaN beam score, makes the whole group an error group (no output);
* a beam score of -inf is allowed (a dead beam): its candidates score -inf
  and rank after every finite candidate.

Test infrastructure only: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline leg may import it.
"""

import math

import numpy as np

from .sampler import logits_to_f64

GROUP_OK = 0
GROUP_BAD_SCORE = 1
GROUP_NONFINITE = 2


def log_softmax64(row):
    """log p of one logit row in float64 (temperature 1)."""
    z = logits_to_f64(row)
    m = np.max(z)
    return z - m - math.log(float(np.sum(np.exp(z - m))))


def candidates(logits, scores):
    """All (score, flat index) candidates of one group: beams x V."""
    out = []
    for b in range(logits.shape[0]):
        lp = log_softmax64(logits[b])
        for t in range(lp.size):
            out.append((float(scores[b]) + float(lp[t]), b * lp.size + t))
    return out


def select_group(logits, scores, width):
    """The `width` best candidates of one group.

    logits: [W, V]; scores: [W] float64.  Returns a dict: parent, token, score
    (lists of `width`), status, and margin (the gap between the last kept and
    the first dropped candidate score, for the parity band).
    """
    logits = np.asarray(logits)
    W, V = logits.shape
    res = {"parent": [-1] * width, "token": [-1] * width, "score": [math.nan] * width,
           "status": GROUP_OK, "margin": math.inf}
    if any(math.isnan(float(s)) for s in scores):
        res["status"] = GROUP_BAD_SCORE
        return res
    for b in range(W):
        if not math.isfinite(float(np.max(logits_to_f64(logits[b])))):
            res["status"] = GROUP_NONFINITE
            return res
    cand = candidates(logits, scores)
    cand.sort(key=lambda c: c[1])                  # appended order: flat index
    cand.sort(key=lambda c: c[0], reverse=True)    # stable: equal scores keep it
    for j in range(min(width, len(cand))):      # ranks past beams x V stay -1 / NaN
        s, flat = cand[j]
        res["parent"][j] = flat // V
        res["token"][j] = flat % V
        res["score"][j] = s
    if len(cand) > width:
        res["margin"] = abs(cand[width - 1][0] - cand[width][0])
    return res


def beam_step(logits, scores, width=None, groups=None):
    """select_group over [G, W, V] logits and [G, W] scores (width W by default)."""
    logits = np.asarray(logits)
    scores = np.asarray(scores, dtype=np.float64)
    G, W, _ = logits.shape
    width = W if width is None else width
    if groups is None:
        groups = range(G)
    out = []
    for g in groups:
        r = select_group(logits[g], scores[g], width)
        r["group"] = int(g)
        out.append(r)
    return out
