"""Benchmark of the sampler and the speculative verifier on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smp|reference]

One step = one smp_sample call on the large-vocabulary batch (B=256,
V=128256, bf16 Zipf-headed logits; half the rows min-p 0.1, a quarter greedy,
a quarter T=0.7 with top-k 40) followed by one smp_spec_verify call on the
verify batch (B=32, K=4, V=32000, fp32).  Inputs are resident in HBM and
rotate over enough copies that every call reads logits that are not in L2.
The K timed steps are replayed from a CUDA graph and timed with CUDA events.

`value` is sampled rows per second of sampler time; the verifier's emitted
tokens per second, the roofline of the sampler kernel, an end-to-end number
through host buffers, the clocks seen during the timed region and the oracle's
own rate on the host cores are reported beside it, on one JSON line.

--impl reference times the fp64 oracle instead, on bounded samples of the
same workload, on the host cores.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sampled rows/s and HBM GB/s (% of peak) at B=256,V=128256 bf16; verify tok/s"
UNIT = "rows/s"
WORKLOAD = "large_vocab"
WORKLOAD_DESC = ("large_vocab: B=256, V=128256, bf16 logits log(Zipf s=1.1) over a seeded per-row "
                 "permutation + N(0, 0.5^2); rows b%4 in {0,1}: min_p=0.1 T=1, b%4==2: greedy, "
                 "b%4==3: T=0.7 top_k=40; Philox seed 0")
VERIFY_DESC = "verify: B=32, K=4, V=32000, fp32; q = G[:, :4], p = G + N(0,1), G ~ N(0, 2^2)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "sample_kernel_large_vocab.md")
KERNEL_SOURCES = ["common.cuh", "row_ops.cuh", "select.cuh", "general.cuh", "sample.cu", "exp_table.h"]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, device=None):
    """The largest `value` over the ranks of the default process group (the
    value itself when there is none): the job takes as long as its slowest
    rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, seconds):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank / seconds


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            data = json.load(fh)
        return float(data["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "spec_verify_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the source."""
    try:
        with open(PROFILE_SUMMARY) as fh:
            text = fh.read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha") != kernel_source_sha():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def oracle_rate(batch, seconds, start_row=0):
    """Rows per second of the fp64 oracle on this process's host core."""
    from oracle import sampler as osam
    done = 0
    t0 = time.perf_counter()
    rows = []
    b = start_row
    while time.perf_counter() - t0 < seconds or done == 0:
        osam.sample(batch.values, batch.params, batch.seed, batch.offset, rows=[b])
        rows.append(b)
        done += 1
        b = (b + 1) % batch.data.shape[0]
    elapsed = time.perf_counter() - t0
    return done / elapsed, done, elapsed


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from spec_verify_gb300 import workloads
    batch = workloads.sampler_workload(WORKLOAD)
    rows_per_step = 4
    from oracle import sampler as osam

    def step(i):
        base = (i * rows_per_step) % batch.data.shape[0]
        osam.sample(batch.values, batch.params, batch.seed, batch.offset,
                    rows=list(range(base, base + rows_per_step)))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    elapsed = time.perf_counter() - t0
    value = rows_per_step * args.steps / elapsed
    sample = f"{rows_per_step} rows of the {WORKLOAD} batch per step, fp64 numpy oracle, one core"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from spec_verify_gb300 import binding
    from spec_verify_gb300 import build as smp_build
    from spec_verify_gb300 import workloads

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    smp_build.build()
    binding.load()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------- inputs, resident in HBM, rotated past L2
    batch = workloads.sampler_workload(WORKLOAD)
    B, V = batch.data.shape
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 2**20))
    sample_bytes = batch.data.nbytes
    n_copies = max(4, math.ceil(4 * l2 / sample_bytes))
    host = torch.from_numpy(batch.data.view(np.int16)).view(torch.bfloat16)
    logits = [host.to(dev) for _ in range(n_copies)]
    params = binding.params_to_device(batch.params, dev)
    out_ids = torch.empty(B, dtype=torch.int32, device=dev)
    out_probs = torch.empty(B, dtype=torch.float32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    seed = rank   # each rank samples its own rows (weak scaling, no collective)

    vb = workloads.verify_workload()
    vB, vK, vV = vb.shape
    v_bytes = vb.p.nbytes + vb.q.nbytes
    v_copies = max(4, math.ceil(4 * l2 / v_bytes))
    p_dev = [torch.from_numpy(vb.p).to(dev) for _ in range(v_copies)]
    q_dev = [torch.from_numpy(vb.q).to(dev) for _ in range(v_copies)]
    d, _, _ = binding.sample(q_dev[0].view(vB * vK, vV), workloads.make_params(vB * vK), vb.draft_seed,
                             vb.draft_offset)
    drafts = d.view(vB, vK).contiguous()
    ws = torch.empty(binding.spec_verify_workspace_bytes(vB, vK), dtype=torch.uint8, device=dev)
    v_acc = torch.empty(vB, dtype=torch.int32, device=dev)
    v_ids = torch.empty(vB, vK + 1, dtype=torch.int32, device=dev)
    v_status = torch.empty(1, dtype=torch.int32, device=dev)

    def sampler_call(i):
        binding.sample(logits[i % n_copies], params, seed, i, out_ids, out_probs, status)

    def sampler_kernel_only(i):   # no status word: sample_kernel alone, for the roofline
        binding.sample(logits[i % n_copies], params, seed, i, out_ids, out_probs, False)

    def verify_call(i):
        binding.spec_verify(p_dev[i % v_copies], q_dev[i % v_copies], drafts, seed, i, ws, v_acc, v_ids,
                            v_status)

    # Verifier variants on the same batch: temperature, greedy, filters (each
    # with drafts drawn from q under the same knobs, by the CUDA sampler).
    variant_knobs = {"temperature_0.8": dict(temperature=0.8), "greedy": dict(greedy=1),
                     "top_k40_top_p0.9_T0.8": dict(temperature=0.8, top_k=40, top_p=0.9),
                     "alpha_T1": dict()}   # T = 1, and the acceptance rates of every position
    v_alpha = torch.empty(vB, vK, dtype=torch.float32, device=dev)
    variants = {}

    def variant_call(name):
        vprm, vdrafts, _ = variants[name]

        def call(i):
            binding.spec_verify_params(p_dev[i % v_copies], q_dev[i % v_copies], vdrafts, vprm, seed, i, ws,
                                       v_acc, v_ids, v_status, out_alpha=v_alpha if name == "alpha_T1" else None)
        return call

    # warm-up (also sets kernel attributes before any capture)
    for i in range(max(args.warmup, 3)):
        sampler_call(i)
        verify_call(i)
    torch.cuda.synchronize()
    assert int(status.cpu()[0]) == 0 and int(v_status.cpu()[0]) == 0

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(args.steps):
                    fn(i)
        torch.cuda.current_stream().wait_stream(s)
        return g

    g_step = capture(lambda i: (sampler_call(i), verify_call(i)))
    g_samp = capture(sampler_call)
    g_kern = capture(sampler_kernel_only)
    g_ver = capture(verify_call)

    def timed(graph, reps):
        for _ in range(reps):       # warm replays
            graph.replay()
        barrier()
        stream = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    with ClockSampler(local) as clocks:
        step_ms = timed(g_step, max(1, args.warmup // max(1, args.steps)))
        samp_ms = timed(g_samp, 1)
        kern_ms = timed(g_kern, 1)
        ver_ms = timed(g_ver, 1)
    clock_info = clocks.summary()
    acc_mean = float(v_acc.float().mean().item())   # accepted lengths of the plain verifier's last call

    # Verifier variants, set up and timed after the headline graphs.
    for name, knobs in variant_knobs.items():
        vprm = binding.params_to_device(workloads.make_params(vB, **knobs), dev)
        dprm = workloads.make_params(vB * vK, **knobs)
        dv, _, _ = binding.sample(q_dev[0].view(vB * vK, vV), dprm, vb.draft_seed, vb.draft_offset)
        variants[name] = (vprm, dv.view(vB, vK).contiguous(), knobs)
    var_ms = {}
    for name in variants:
        call = variant_call(name)
        for i in range(max(args.warmup, 3)):
            call(i)
        torch.cuda.synchronize()
        assert int(v_status.cpu()[0]) == 0
        g = capture(call)
        ms = timed(g, 1)
        var_ms[name] = (ms, float(v_acc.float().mean().item()))   # accepted lengths of the last call
        del g
    # Sampler with the logit pre-pass on the headline batch: repetition
    # penalty over 64 recent tokens, with and without a constraint mask.
    allowed_np, history_np, penalty_np = workloads.prepass_inputs(batch.values, seed=1, mask_density=(0.8, 1.0))
    allowed_np[-1] = allowed_np[-2]   # no error row in the timed batch
    allowed_dev = torch.from_numpy(allowed_np.view(np.int32)).to(dev)
    history_dev = torch.from_numpy(history_np).to(dev)
    penalty_dev = torch.from_numpy(penalty_np).to(dev)
    sampler_variants = {}
    for name, use_mask in (("penalty", False), ("penalty_and_mask", True)):
        def pcall(i, use_mask=use_mask):
            binding.sample_processed(logits[i % n_copies], params, seed, i, allowed_dev if use_mask else None,
                                     history_dev, penalty_dev, out_ids, out_probs, status)
        for i in range(max(args.warmup, 3)):
            pcall(i)
        torch.cuda.synchronize()
        assert int(status.cpu()[0]) == 0
        g = capture(pcall)
        us = 1000.0 * timed(g, 1) / args.steps
        del g
        nbytes = sample_bytes + (allowed_np.nbytes if use_mask else 0) + history_np.nbytes + penalty_np.nbytes
        sampler_variants[name] = {"us_per_call": us, "rows_per_s": job_rate(B, world, us * 1e-6),
                                  "bytes_per_call": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9}

    # The same through the in-place pre-pass: smp_logit_prepass, then
    # smp_sample (the copies are modified in place; the penalty compounds
    # over replays on the same copy, which changes no byte count).
    for name, use_mask in (("inplace_penalty_then_sample", False), ("inplace_penalty_and_mask_then_sample", True)):
        def icall(i, use_mask=use_mask):
            binding.logit_prepass(logits[i % n_copies], allowed_dev if use_mask else None, history_dev,
                                  penalty_dev, status)
            binding.sample(logits[i % n_copies], params, seed, i, out_ids, out_probs, status)
        for i in range(max(args.warmup, 3)):
            icall(i)
        torch.cuda.synchronize()
        g = capture(icall)
        us = 1000.0 * timed(g, 1) / args.steps
        del g
        nbytes = sample_bytes + (allowed_np.nbytes if use_mask else 0) + history_np.nbytes + penalty_np.nbytes
        sampler_variants[name] = {"us_per_call": us, "rows_per_s": job_rate(B, world, us * 1e-6),
                                  "bytes_per_call": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9}

    # One beam-search step: 8 requests x 4 beams over the large vocabulary
    # (bf16, Zipf-headed logits), the 4 best candidates of each request.
    bG, bW, bwidth = 8, 4, 4
    brng = np.random.default_rng(3000)
    bz = workloads.f32_to_bf16_bits(workloads.zipf_logits_f32(brng, bG * bW, V)).reshape(bG, bW, V)
    b_bytes = bz.nbytes
    b_copies = max(4, math.ceil(4 * l2 / b_bytes))
    b_host = torch.from_numpy(bz.view(np.int16)).view(torch.bfloat16)
    b_dev = [b_host.to(dev) for _ in range(b_copies)]
    b_scores = torch.from_numpy(-brng.uniform(0, 12, (bG, bW))).to(dev)
    b_ws = torch.empty(max(8, int(binding.load().smp_beam_topk_workspace_bytes(bG, bW, bwidth))),
                       dtype=torch.uint8, device=dev)
    b_par = torch.empty(bG, bwidth, dtype=torch.int32, device=dev)
    b_tok = torch.empty(bG, bwidth, dtype=torch.int32, device=dev)
    b_sc = torch.empty(bG, bwidth, dtype=torch.float64, device=dev)

    def bcall(i):
        binding.beam_topk(b_dev[i % b_copies], b_scores, bwidth, b_ws, b_par, b_tok, b_sc, status)
    for i in range(max(args.warmup, 3)):
        bcall(i)
    torch.cuda.synchronize()
    assert int(status.cpu()[0]) == 0
    g = capture(bcall)
    b_us = 1000.0 * timed(g, 1) / args.steps
    del g
    beam_line = {"workload": f"{bG} requests x {bW} beams x V={V} bf16 (Zipf-headed), width {bwidth}",
                 "us_per_call": b_us, "steps_per_s": world / (b_us * 1e-6), "bytes_per_call": b_bytes,
                 "gbs": b_bytes / (b_us * 1e-6) / 1e9,
                 "l2": f"inputs rotate over {b_copies} copies ({b_copies * b_bytes / 1e6:.0f} MB)"}

    verify_variants = {}
    for name, (ms, accepted) in var_ms.items():
        us = 1000.0 * ms / args.steps
        nbytes = vb.p.nbytes if "greedy" in name else v_bytes   # greedy reads no draft row
        verify_variants[name] = {"us_per_call": us, "mean_accepted": accepted,
                                 "tok_s": world * vB * (accepted + 1.0) / (us * 1e-6),
                                 "bytes_per_call": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9,
                                 "knobs": variants[name][2]}

    # per step: clear_status_kernel + sample_kernel, verify_pos_kernel (which clears the
    # verifier's status word) + verify_resolve_kernel
    gpu_launches = args.steps * 4
    samp_us = 1000.0 * samp_ms / args.steps
    kern_us = 1000.0 * kern_ms / args.steps
    ver_us = 1000.0 * ver_ms / args.steps
    rows_per_s = job_rate(B, world, samp_us * 1e-6)
    verify_tok_s = world * vB * (acc_mean + 1.0) / (ver_us * 1e-6)

    # roofline of the sampler kernel: logits read once, ids + probs written, params read
    alg_bytes = B * V * 2 + B * 8 + B * 20
    achieved = alg_bytes / (kern_us * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(),
                "kernel": "sample_kernel", "kernel_us_per_launch": kern_us,
                "timing": "K back-to-back sample_kernel launches (no status word) in one CUDA graph",
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                "algorithmic_bytes_per_launch": alg_bytes}

    # ---------------- end to end through the public API with host buffers
    pinned = host.pin_memory()
    params_host = torch.from_numpy(batch.params.view(np.uint8).copy()).pin_memory()
    ids_host = torch.empty(B, dtype=torch.int32).pin_memory()
    probs_host = torch.empty(B, dtype=torch.float32).pin_memory()
    # Two input buffers: step i's copy (on its own stream) overlaps step
    # i - 1's sampler call; a buffer is refilled only after the call that read
    # it has finished.  Every step still copies its whole input.
    dev_in = [torch.empty_like(logits[0]) for _ in range(2)]
    dev_params = [torch.empty_like(params) for _ in range(2)]
    copy_stream = torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    for ev in freed:
        ev.record(compute)
    e2e_steps = max(3, args.steps)

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(freed[k])
            dev_in[k].copy_(pinned, non_blocking=True)
            dev_params[k].copy_(params_host, non_blocking=True)
            copied[k].record(copy_stream)
        compute.wait_event(copied[k])
        binding.sample(dev_in[k], dev_params[k], seed, i, out_ids, out_probs, status)
        freed[k].record(compute)
        ids_host.copy_(out_ids, non_blocking=True)
        probs_host.copy_(out_probs, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    copy_stream.wait_stream(compute)   # the first copy starts after e0
    for i in range(e2e_steps):
        e2e_step(i)
    compute.wait_stream(copy_stream)
    e1.record()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e = {"value": job_rate(B * e2e_steps, world, e2e_ms * 1e-3), "unit": UNIT,
           "h2d_bytes_per_step": sample_bytes + batch.params.nbytes, "d2h_bytes_per_step": B * 8,
           "what": "pinned host logits+params -> device copy (own stream, two buffers: overlaps the previous step's call), smp_sample, ids+probs -> host, per step"}

    # ---------------- oracle on the host cores (rank 0, N = 1 only)
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows_done, secs = oracle_rate(batch, args.cpu_seconds)
        cpu_baseline = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                        "sample": f"{rows_done} rows of the {WORKLOAD} batch in {secs:.1f} s, fp64 numpy oracle"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": rows_per_s, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "batch": B, "vocab": V, "logits_dtype": "bf16",
                       "verify_workload": VERIFY_DESC,
                       "l2": f"inputs rotate over {n_copies} sampler copies ({n_copies * sample_bytes / 1e6:.0f} MB) "
                             f"and {v_copies} verify copies; L2 {l2 / 1e6:.0f} MB",
                       "timing": "K steps captured in one CUDA graph, CUDA events on the launching stream",
                       "parallelism": f"dp{world} (rows independent, no collective)"},
            "sampler_us_per_call": samp_us,
            "sample_kernel_us": kern_us,
            "hbm_gbs": achieved,
            "sampler_variants": sampler_variants,
            "beam_step": beam_line,
            "pct_of_measured_hbm": 100.0 * achieved / peak,
            "pct_of_8tbs_nominal": 100.0 * achieved / NOMINAL_HBM_GBS,
            "verify": {"tok_s": verify_tok_s, "us_per_call": ver_us, "mean_accepted": acc_mean,
                       "bytes_per_call": v_bytes, "gbs": v_bytes / (ver_us * 1e-6) / 1e9,
                       "variants": verify_variants},
            "roofline": roofline,
            "cpu_baseline": cpu_baseline,
            "e2e": e2e,
            "gpu_launches": gpu_launches,
            "clocks": clock_info,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["smp", "reference"], default="smp")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
