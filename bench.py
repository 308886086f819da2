"""Benchmark of the sampler and the speculative verifier on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smp|reference]

One step = one smp_sample call on the large-vocabulary batch (B=256,
V=128256, bf16 Zipf-headed logits; half the rows min-p 0.1, a quarter greedy,
a quarter T=0.7 with top-k 40) followed by one smp_spec_verify call on the
verify batch (B=32, K=4, V=32000, fp32).  Inputs are resident in HBM and
rotate over enough copies that no call finds its logits in L2.  The K steps
are captured in one CUDA graph; the graph is replayed at least 10 times, each
replay timed with CUDA events on the launching stream between a barrier and a
device synchronisation, and the median replay (the best beside it) gives the
per-call time.

With N GPUs (torchrun, one process per GPU) the job is one batch of N x 256
rows split by rows: rank r takes rows [256 r, 256 (r + 1)) and passes 256 r as
the row base of its Philox counters, so the tokens do not depend on the split
and no collective runs on the data path (weak scaling); the time is the
maximum over ranks.

`value` is sampled rows per second of sampler time; the verifier's emitted
tokens per second, the roofline of the sampler kernel, the general-path
workloads (the mixed batch and the wide-nucleus batch), an end-to-end number
through host buffers, the clocks seen during the timed region and the
oracle's own rate on the host cores are reported beside it, on one JSON line.

--impl reference times the fp64 oracle instead, on bounded samples of the
same workload, on all host cores.
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
# The path's arithmetic: binary32 (exponentials as double-float pairs of
# binary32, comparisons); masses are summed as exact u64 integers.
DTYPE = "f32"
ARITHMETIC = "bf16 logits; exp in double-float (pairs of binary32); u64 fixed-point masses, exact integer sums"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILE_JSON = os.path.join(ROOT, "profiles", "sample_kernel_large_vocab.json")
KERNEL_SOURCES = ["common.cuh", "row_ops.cuh", "select.cuh", "general.cuh", "sample.cu", "exp_table.h", "tma.cuh", "general_bf16.cuh"]
MIN_REPLAYS = 10


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def row_block(rows, rank, world):
    """The contiguous block [lo, hi) of a batch of `rows` rows that rank
    `rank` of `world` takes (sizes differ by at most one)."""
    base, extra = divmod(rows, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


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


def profiled_traffic(path=PROFILE_JSON):
    """DRAM bytes per launch of sample_kernel from the committed ncu capture
    (profiles/*.json, written with the capture), or None when the kernel
    sources have changed since the counters were taken."""
    try:
        with open(path) as fh:
            data = json.load(fh)
    except (OSError, ValueError):
        return None
    if data.get("source_sha") != kernel_source_sha():
        return None
    try:
        return float(data["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
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


# ---------------------------------------------------------------- the oracle on the host cores

def cpu_baseline(batch, seconds):
    """The fp64 oracle on all host cores and on one core (spawned worker
    processes, so nothing of the GPU process competes with them), each over
    whole passes of the batch sized to about `seconds`.  Returns the
    cpu_baseline object of the JSON line."""
    from oracle import pool
    B = batch.data.shape[0]
    cores = pool.default_procs()
    probe, _, _ = pool.sampler_rate(batch.values, batch.params, batch.seed, batch.offset, range(B), 1)
    passes_1 = max(1, int(round(seconds * probe / B)))
    passes_all = max(1, int(round(seconds * probe * cores / B)))
    rate_1, n_1, s_1 = pool.sampler_rate(batch.values, batch.params, batch.seed, batch.offset,
                                         list(range(B)) * passes_1, 1)
    rate_all, n_all, s_all = pool.sampler_rate(batch.values, batch.params, batch.seed, batch.offset,
                                               list(range(B)) * passes_all, cores)
    return {"value": rate_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"{n_all} rows ({passes_all} passes over the {WORKLOAD} batch) in {s_all:.1f} s on "
                       f"{cores} worker processes, one per core; {n_1} rows in {s_1:.1f} s on one; fp64 numpy "
                       f"oracle"),
            "cores_all": cores, "rows_per_s_all": rate_all, "rows_per_s_1": rate_1}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import multiprocessing as mp

    from oracle import pool
    from spec_verify_gb300 import workloads
    batch = workloads.sampler_workload(WORKLOAD)
    B = batch.data.shape[0]
    cores = pool.default_procs()
    rows_per_step = 4 * cores
    handles, specs = pool._share({"values": batch.values, "params": batch.params})
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(processes=cores, initializer=pool._attach, initargs=(specs,)) as workers:
            def step(i):
                base = (i * rows_per_step) % B
                rows = [(base + j) % B for j in range(rows_per_step)]
                chunks = [rows[j::cores] for j in range(cores)]
                workers.map(pool._timed_sample_chunk, [(c, batch.seed, batch.offset) for c in chunks],
                            chunksize=1)

            for i in range(args.warmup):
                step(i)
            t0 = time.perf_counter()
            for i in range(args.steps):
                step(args.warmup + i)
            elapsed = time.perf_counter() - t0
    finally:
        for h in handles:
            h.close()
            h.unlink()
    value = rows_per_step * args.steps / elapsed
    sample = (f"{rows_per_step} rows of the {WORKLOAD} batch per step (cycling through it), fp64 numpy oracle "
              f"on {cores} worker processes, one per host core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- the GPU arm

def run_gpu(args):
    import torch
    import torch.distributed as dist

    from spec_verify_gb300 import binding
    from spec_verify_gb300 import build as smp_build
    from spec_verify_gb300 import workloads

    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one process per GPU with "
                         f"torchrun --nproc-per-node {args.gpus}")
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

    steps = args.steps
    replays = max(MIN_REPLAYS, args.replays)

    # ---------------- inputs, resident in HBM, rotated past L2
    batch = workloads.sampler_workload(WORKLOAD)
    B, V = batch.data.shape
    row_base, _ = row_block(world * B, rank, world)     # this rank's rows of the N x B job
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 2**20))
    sample_bytes = batch.data.nbytes

    def copies(nbytes):
        return max(4, math.ceil(4 * l2 / nbytes))

    n_copies = copies(sample_bytes)
    host = torch.from_numpy(batch.data.view(np.int16)).view(torch.bfloat16)
    logits = [host.to(dev) for _ in range(n_copies)]
    params = binding.params_to_device(batch.params, dev)
    out_ids = torch.empty(B, dtype=torch.int32, device=dev)
    out_probs = torch.empty(B, dtype=torch.float32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    seed = batch.seed

    vb = workloads.verify_workload()
    vB, vK, vV = vb.shape
    v_base, _ = row_block(world * vB, rank, world)
    v_bytes = vb.p.nbytes + vb.q.nbytes
    v_copies = copies(v_bytes)
    p_dev = [torch.from_numpy(vb.p).to(dev) for _ in range(v_copies)]
    q_dev = [torch.from_numpy(vb.q).to(dev) for _ in range(v_copies)]
    d, _, _ = binding.sample(q_dev[0].view(vB * vK, vV), workloads.make_params(vB * vK), vb.draft_seed,
                             vb.draft_offset)
    drafts = d.view(vB, vK).contiguous()
    ws = torch.zeros(binding.spec_verify_workspace_bytes(vB, vK), dtype=torch.uint8, device=dev)
    v_acc = torch.empty(vB, dtype=torch.int32, device=dev)
    v_ids = torch.empty(vB, vK + 1, dtype=torch.int32, device=dev)
    v_status = torch.empty(1, dtype=torch.int32, device=dev)

    def sampler_call(i):
        binding.sample_rows(logits[i % n_copies], params, seed, i, row_base, out_ids=out_ids, out_probs=out_probs,
                            status=status)

    def sampler_kernel_only(i):   # no status word: sample_kernel alone, for the roofline
        binding.sample_rows(logits[i % n_copies], params, seed, i, row_base, out_ids=out_ids, out_probs=out_probs,
                            status=False)

    def sampler_warm_l2(i):       # one copy, resident in L2 after the first call
        binding.sample_rows(logits[0], params, seed, i, row_base, out_ids=out_ids, out_probs=out_probs,
                            status=False)

    def verify_call(i):
        binding.spec_verify_rows(p_dev[i % v_copies], q_dev[i % v_copies], drafts, None, vb.seed, i, v_base,
                                 workspace=ws, out_accepted=v_acc, out_ids=v_ids, status=v_status)

    # warm-up (also sets kernel attributes before any capture)
    for i in range(args.warmup):
        sampler_call(i)
        verify_call(i)
    torch.cuda.synchronize()
    assert int(status.cpu()[0]) == 0 and int(v_status.cpu()[0]) == 0

    def capture(fn, n=steps):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    fn(i)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def timed(graph, calls=steps):
        """Per-call microseconds of a graph of `calls` calls: (median, best)
        over `replays` replays, each between a barrier and a synchronize,
        maximum over ranks."""
        graph.replay()               # warm replay
        stream = torch.cuda.current_stream()
        times = []
        for _ in range(replays):
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            barrier()
            times.append(max_over_ranks(e0.elapsed_time(e1), dev))
        return 1000.0 * statistics.median(times) / calls, 1000.0 * min(times) / calls

    g_step = capture(lambda i: (sampler_call(i), verify_call(i)))
    g_samp = capture(sampler_call)
    g_kern = capture(sampler_kernel_only)
    g_warm = capture(sampler_warm_l2)
    g_ver = capture(verify_call)

    with ClockSampler(local) as clocks:
        step_us, step_best = timed(g_step)
        samp_us, samp_best = timed(g_samp)
        kern_us, kern_best = timed(g_kern)
        warm_us, warm_best = timed(g_warm)
        ver_us, ver_best = timed(g_ver)
    clock_info = clocks.summary()
    acc_mean = float(v_acc.float().mean().item())   # accepted lengths of the plain verifier's last call
    del g_step, g_samp, g_kern, g_warm, g_ver

    def graph_line(fn, nbytes, units, calls=steps):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        g = capture(fn, calls)
        med, best = timed(g, calls)
        del g
        return {"us_per_call": med, "us_best": best, "units_per_s": job_rate(units, world, med * 1e-6),
                "bytes_per_call": nbytes, "gbs": nbytes / (med * 1e-6) / 1e9}

    peak, peak_kind = measured_peaks()

    # ---------------- the general path: the mixed batch and the wide nucleus
    general = {}
    for name in ("mixed", "flat_nucleus"):
        gb = workloads.sampler_workload(name)
        gB, gV = gb.data.shape
        g_host = torch.from_numpy(gb.data.view(np.int16)).view(torch.bfloat16)
        g_n = copies(gb.data.nbytes)
        g_dev = [g_host.to(dev) for _ in range(g_n)]
        g_prm = binding.params_to_device(gb.params, dev)
        g_ids = torch.empty(gB, dtype=torch.int32, device=dev)
        g_probs = torch.empty(gB, dtype=torch.float32, device=dev)
        g_base, _ = row_block(world * gB, rank, world)

        def gcall(i, g_dev=g_dev, g_prm=g_prm, g_ids=g_ids, g_probs=g_probs, g_base=g_base, g_n=g_n):
            binding.sample_rows(g_dev[i % g_n], g_prm, gb.seed, i, g_base, out_ids=g_ids, out_probs=g_probs,
                                status=status)

        nbytes = gB * (gV * 2 + 28)
        line = graph_line(gcall, nbytes, gB, calls=min(steps, 50))
        assert int(status.cpu()[0]) == 0
        line["rows_per_s"] = line.pop("units_per_s")
        line["frac_of_measured_hbm"] = line["gbs"] / peak
        line["workload"] = f"{name}: B={gB}, V={gV}, bf16"
        line["l2"] = f"inputs rotate over {g_n} copies ({g_n * gb.data.nbytes / 1e6:.0f} MB)"
        general[name] = line
        del g_dev
        torch.cuda.empty_cache()

    # ---------------- verifier variants on the same batch
    variant_knobs = {"temperature_0.8": dict(temperature=0.8), "greedy": dict(greedy=1),
                     "top_k40_top_p0.9_T0.8": dict(temperature=0.8, top_k=40, top_p=0.9),
                     "alpha_T1": dict()}   # T = 1, and the acceptance rates of every position
    v_alpha = torch.empty(vB, vK, dtype=torch.float32, device=dev)
    verify_variants = {}
    for name, knobs in variant_knobs.items():
        vprm = binding.params_to_device(workloads.make_params(vB, **knobs), dev)
        dprm = workloads.make_params(vB * vK, **knobs)
        dv, _, _ = binding.sample(q_dev[0].view(vB * vK, vV), dprm, vb.draft_seed, vb.draft_offset)
        vdrafts = dv.view(vB, vK).contiguous()

        def vcall(i, vprm=vprm, vdrafts=vdrafts, name=name):
            binding.spec_verify_rows(p_dev[i % v_copies], q_dev[i % v_copies], vdrafts, vprm, vb.seed, i, v_base,
                                     workspace=ws, out_accepted=v_acc, out_ids=v_ids, status=v_status,
                                     out_alpha=v_alpha if name == "alpha_T1" else None)

        nbytes = vb.p.nbytes if "greedy" in name else v_bytes   # greedy reads no draft row
        line = graph_line(vcall, nbytes, vB)
        assert int(v_status.cpu()[0]) == 0
        accepted = float(v_acc.float().mean().item())
        line.pop("units_per_s")
        line.update({"mean_accepted": accepted, "tok_s": world * vB * (accepted + 1.0) / (line["us_per_call"] * 1e-6),
                     "knobs": knobs})
        verify_variants[name] = line

    # ---------------- sampler with the logit pre-pass on the headline batch
    allowed_np, history_np, penalty_np = workloads.prepass_inputs(batch.values, seed=1, mask_density=(0.8, 1.0))
    allowed_np[-1] = allowed_np[-2]   # no error row in the timed batch
    allowed_dev = torch.from_numpy(allowed_np.view(np.int32)).to(dev)
    history_dev = torch.from_numpy(history_np).to(dev)
    penalty_dev = torch.from_numpy(penalty_np).to(dev)
    sampler_variants = {}
    for name, use_mask in (("penalty", False), ("penalty_and_mask", True)):
        def pcall(i, use_mask=use_mask):
            binding.sample_rows(logits[i % n_copies], params, seed, i, row_base,
                                allowed=allowed_dev if use_mask else None, history=history_dev,
                                penalty=penalty_dev, out_ids=out_ids, out_probs=out_probs, status=status)
        nbytes = sample_bytes + (allowed_np.nbytes if use_mask else 0) + history_np.nbytes + penalty_np.nbytes
        line = graph_line(pcall, nbytes, B)
        assert int(status.cpu()[0]) == 0
        line["rows_per_s"] = line.pop("units_per_s")
        sampler_variants[name] = line
    # The same through the in-place pre-pass: smp_logit_prepass, then
    # smp_sample (the copies are modified in place; the penalty compounds
    # over replays on the same copy, which changes no byte count).
    for name, use_mask in (("inplace_penalty_then_sample", False), ("inplace_penalty_and_mask_then_sample", True)):
        def icall(i, use_mask=use_mask):
            binding.logit_prepass(logits[i % n_copies], allowed_dev if use_mask else None, history_dev,
                                  penalty_dev, status)
            binding.sample_rows(logits[i % n_copies], params, seed, i, row_base, out_ids=out_ids,
                                out_probs=out_probs, status=status)
        nbytes = sample_bytes + (allowed_np.nbytes if use_mask else 0) + history_np.nbytes + penalty_np.nbytes
        line = graph_line(icall, nbytes, B)
        line["rows_per_s"] = line.pop("units_per_s")
        sampler_variants[name] = line

    # ---------------- one beam-search step: 8 requests x 4 beams over the large vocabulary
    bG, bW, bwidth = 8, 4, 4
    brng = np.random.default_rng(3000)
    bz = workloads.f32_to_bf16_bits(workloads.zipf_logits_f32(brng, bG * bW, V)).reshape(bG, bW, V)
    b_bytes = bz.nbytes
    b_copies = copies(b_bytes)
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
    beam_line = graph_line(bcall, b_bytes, 1)
    assert int(status.cpu()[0]) == 0
    beam_line["steps_per_s"] = beam_line.pop("units_per_s")
    beam_line["workload"] = f"{bG} requests x {bW} beams x V={V} bf16 (Zipf-headed), width {bwidth}"
    beam_line["l2"] = f"inputs rotate over {b_copies} copies ({b_copies * b_bytes / 1e6:.0f} MB)"
    del b_dev

    # per step: clear_status_kernel + sample_kernel, then the verifier's kernels
    gpu_launches = steps * (2 + binding.VERIFY_LAUNCHES)
    rows_per_s = job_rate(B, world, samp_us * 1e-6)
    verify_tok_s = world * vB * (acc_mean + 1.0) / (ver_us * 1e-6)

    # roofline of the sampler kernel: logits read once, ids + probs written, params read
    alg_bytes = B * V * 2 + B * 8 + B * 20
    achieved = alg_bytes / (kern_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(),
                "kernel": "sample_kernel", "kernel_us_per_launch": kern_us, "kernel_us_best": kern_best,
                "timing": (f"K back-to-back sample_kernel launches (no status word) in one CUDA graph, median of "
                           f"{replays} replays"),
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
    e2e_steps = max(3, steps)

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(freed[k])
            dev_in[k].copy_(pinned, non_blocking=True)
            dev_params[k].copy_(params_host, non_blocking=True)
            copied[k].record(copy_stream)
        compute.wait_event(copied[k])
        binding.sample_rows(dev_in[k], dev_params[k], seed, i, row_base, out_ids=out_ids, out_probs=out_probs,
                            status=status)
        freed[k].record(compute)
        ids_host.copy_(out_ids, non_blocking=True)
        probs_host.copy_(out_probs, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    barrier()
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
           "what": ("pinned host logits+params -> device copy (own stream, two buffers: overlaps the previous "
                    "step's call), smp_sample_rows, ids+probs -> host, per step")}

    # ---------------- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batch, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": rows_per_s, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": step_us / 1000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "batch": B, "vocab": V, "logits_dtype": "bf16",
                       "verify_workload": VERIFY_DESC,
                       "l2": f"inputs rotate over {n_copies} sampler copies ({n_copies * sample_bytes / 1e6:.0f} MB) "
                             f"and {v_copies} verify copies; L2 {l2 / 1e6:.0f} MB",
                       "timing": (f"K steps captured in one CUDA graph, replayed {replays} times, CUDA events on "
                                  f"the launching stream; median replay (best beside it)"),
                       "arithmetic": ARITHMETIC,
                       "parallelism": (f"dp{world}: a batch of {world} x {B} rows split by rows, rank r at row base "
                                       f"{B} r (no collective)")},
            "ms_per_step_best": step_best / 1000.0,
            "sampler_us_per_call": samp_us, "sampler_us_best": samp_best,
            "sample_kernel_us": kern_us, "sample_kernel_us_best": kern_best,
            "warm_l2": {"us_per_call": warm_us, "us_best": warm_best,
                        "what": "sample_kernel on one copy of the batch (L2-resident after the first call)"},
            "hbm_gbs": achieved,
            "pct_of_measured_hbm": 100.0 * achieved / peak,
            "pct_of_8tbs_nominal": 100.0 * achieved / NOMINAL_HBM_GBS,
            "general_path": general,
            "sampler_variants": sampler_variants,
            "beam_step": beam_line,
            "verify": {"tok_s": verify_tok_s, "us_per_call": ver_us, "us_best": ver_best, "mean_accepted": acc_mean,
                       "bytes_per_call": v_bytes, "gbs": v_bytes / (ver_us * 1e-6) / 1e9,
                       "frac_of_measured_hbm": v_bytes / (ver_us * 1e-6) / 1e9 / peak,
                       "variants": verify_variants},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": gpu_launches,
            "clocks": clock_info,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_case(args):
    """One sampler workload by plain calls (no graph), for profilers: W
    untimed calls, then K calls timed together with CUDA events; prints one
    JSON line with the per-call time."""
    import numpy as np
    import torch
    from spec_verify_gb300 import binding, workloads
    binding.load()
    gb = workloads.sampler_workload(args.case)
    B, V = gb.data.shape
    if gb.dtype == "bf16":
        x = torch.from_numpy(gb.data.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        x = torch.from_numpy(gb.data).cuda()
    prm = binding.params_to_device(gb.params, x.device)
    ids = torch.empty(B, dtype=torch.int32, device=x.device)
    probs = torch.empty(B, dtype=torch.float32, device=x.device)
    status = torch.empty(1, dtype=torch.int32, device=x.device)
    for i in range(args.warmup):
        binding.sample_rows(x, prm, gb.seed, i, 0, out_ids=ids, out_probs=probs, status=status)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        binding.sample_rows(x, prm, gb.seed, args.warmup + i, 0, out_ids=ids, out_probs=probs, status=status)
    e1.record()
    torch.cuda.synchronize()
    if int(status.cpu()[0]) != 0:
        raise SystemExit(f"status {int(status.cpu()[0])}")
    print(json.dumps({"case": args.case, "batch": B, "vocab": V, "dtype": gb.dtype, "calls": args.steps,
                      "us_per_call": 1000.0 * e0.elapsed_time(e1) / args.steps,
                      "l2": "one input copy, reused by every call"}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--replays", type=int, default=MIN_REPLAYS, help=f"graph replays timed (at least {MIN_REPLAYS})")
    ap.add_argument("--impl", choices=["smp", "reference"], default="smp")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", choices=["basic", "mixed", "large_vocab", "flat_nucleus"],
                    help="only time plain sampler calls on this workload (for profilers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
