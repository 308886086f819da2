"""Shared helpers for the GPU parity tests: device upload and the comparison
rule between the CUDA path and the oracle.

Rule: kept sets and token ids must be identical, except rows whose oracle
cumulative sum lies within 1e-6 of top_p, whose uniform lies within 1e-6 of a
CDF boundary, whose p_i / p_max lies within 1e-6 of min_p, or (verifier) whose
accept uniform lies within 1e-6 of p/q.  Such rows are excused only if they
are fewer than 1e-4 of the rows compared (so, below 10^4 rows, none).
Probabilities must agree within 1e-5 relative.
"""

import math

import numpy as np

BAND = 1e-6
EXCUSE_FRACTION = 1e-4
PROB_RTOL = 1e-5


def torch():
    import torch as _t
    return _t


def device_logits(data, dtype):
    """Upload a numpy logits array (float32 values or bf16 bit patterns)."""
    t = torch()
    if dtype == "bf16":
        host = t.from_numpy(np.ascontiguousarray(data).view(np.int16)).view(t.bfloat16)
    else:
        host = t.from_numpy(np.ascontiguousarray(data, dtype=np.float32))
    return host.cuda().contiguous()


class Verdict:
    def __init__(self):
        self.compared = 0
        self.excused = []
        self.failed = []
        self.prob_failures = []

    def check(self):
        assert not self.failed, f"{len(self.failed)} mismatching rows outside the band: {self.failed[:8]}"
        budget = math.floor(EXCUSE_FRACTION * self.compared)
        assert len(self.excused) <= budget, f"{len(self.excused)} in-band mismatches (budget {budget}): {self.excused[:8]}"
        assert not self.prob_failures, f"probabilities off: {self.prob_failures[:8]}"


def compare_sampler(oracle_rows, gpu_ids, gpu_probs):
    """Compare oracle.sampler.sample results with GPU ids / probs (numpy)."""
    v = Verdict()
    for res in oracle_rows:
        b = res["row"]
        v.compared += 1
        g = int(gpu_ids[b])
        if g != res["token"]:
            margin = min(res["topp_margin"], res["draw_margin"], res["minp_margin"])
            entry = (b, g, res["token"], margin)
            (v.excused if margin < BAND else v.failed).append(entry)
            continue
        if res["token"] < 0:
            if not math.isnan(float(gpu_probs[b])):
                v.prob_failures.append((b, float(gpu_probs[b]), "nan expected"))
            continue
        want, got = res["prob"], float(gpu_probs[b])
        if not abs(got - want) <= PROB_RTOL * abs(want):
            v.prob_failures.append((b, got, want))
    return v


def compare_verify(oracle_rows, gpu_acc, gpu_ids):
    v = Verdict()
    for res in oracle_rows:
        b = res["row"]
        v.compared += 1
        same = int(gpu_acc[b]) == res["accepted"] and list(map(int, gpu_ids[b])) == res["ids"]
        if not same:
            margin = min(res["accept_margin"], res["draw_margin"], res.get("filter_margin", math.inf))
            entry = (b, int(gpu_acc[b]), list(map(int, gpu_ids[b])), res["accepted"], res["ids"], margin)
            (v.excused if margin < BAND else v.failed).append(entry)
    return v
