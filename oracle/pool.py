"""Runs the oracle over the rows of a batch on several host cores (test
infrastructure, like the rest of this package).

The per-row functions of oracle.sampler and oracle.verify are unchanged; this
module only splits a batch's rows into chunks and hands them to worker
processes.  The logits are placed once in shared memory, so no worker copies
them.  Workers are started with the "spawn" method: a process forked from one
that has already used the GPU can hang, and spawn works whether or not it has.

Results are identical to one call of the per-row function over the same rows
(each row draws its own uniforms from the Philox counter; nothing is shared
between rows).
"""

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

from . import sampler, verify

_ARRAYS = {}
_SHMS = []


def default_procs():
    """Host cores available to this process."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _share(arrays):
    """Copy named numpy arrays into shared memory; returns (handles, specs)."""
    handles, specs = [], {}
    for name, arr in arrays.items():
        if arr is None:
            specs[name] = None
            continue
        arr = np.ascontiguousarray(arr)
        shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
        np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
        handles.append(shm)
        specs[name] = (shm.name, arr.shape, arr.dtype)
    return handles, specs


def _attach(specs):
    _ARRAYS.clear()
    for name, spec in specs.items():
        if spec is None:
            _ARRAYS[name] = None
            continue
        shm_name, shape, dt = spec
        shm = shared_memory.SharedMemory(name=shm_name)
        _SHMS.append(shm)
        _ARRAYS[name] = np.ndarray(shape, dtype=np.dtype(dt), buffer=shm.buf)


def _sample_chunk(job):
    rows, seed, offset, row_base = job
    return sampler.sample(_ARRAYS["values"], _ARRAYS["params"], seed, offset, rows=rows, row_base=row_base)


def _verify_chunk(job):
    rows, seed, offset, row_base, extra = job
    return verify.spec_verify(_ARRAYS["p"], _ARRAYS["q"], _ARRAYS["drafts"], seed, offset, rows=rows,
                              params=_ARRAYS["params"], row_base=row_base, **extra)


def _chunks(rows, procs, per_chunk=None):
    rows = list(rows)
    if per_chunk is None:
        per_chunk = max(1, len(rows) // (4 * procs))
    return [rows[i:i + per_chunk] for i in range(0, len(rows), per_chunk)]


def _run(arrays, fn, jobs, procs):
    handles, specs = _share(arrays)
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(processes=procs, initializer=_attach, initargs=(specs,)) as pool:
            parts = pool.map(fn, jobs, chunksize=1)
    finally:
        for h in handles:
            h.close()
            h.unlink()
    return [r for part in parts for r in part]


def sample_parallel(values, params, seed, offset, rows=None, row_base=0, procs=None):
    """oracle.sampler.sample over `rows` (default: all), split across procs workers."""
    procs = procs or default_procs()
    rows = range(np.asarray(values).shape[0]) if rows is None else rows
    jobs = [(c, seed, offset, row_base) for c in _chunks(rows, procs)]
    return _run({"values": values, "params": params}, _sample_chunk, jobs, procs)


def spec_verify_parallel(p_values, q_values, drafts, seed, offset, rows=None, params=None, row_base=0, procs=None,
                         **extra):
    """oracle.verify.spec_verify over `rows` (default: all), split across procs
    workers; `extra` goes to spec_verify (temperature, greedy, alpha)."""
    procs = procs or default_procs()
    rows = range(np.asarray(p_values).shape[0]) if rows is None else rows
    jobs = [(c, seed, offset, row_base, extra) for c in _chunks(rows, procs)]
    return _run({"p": p_values, "q": q_values, "drafts": drafts, "params": params}, _verify_chunk, jobs, procs)


def _timed_sample_chunk(job):
    rows, seed, offset = job
    t0 = time.perf_counter()
    sampler.sample(_ARRAYS["values"], _ARRAYS["params"], seed, offset, rows=rows)
    return len(rows), time.perf_counter() - t0


def sampler_rate(values, params, seed, offset, rows, procs):
    """Rows per second of the oracle sampler over `rows` on `procs` worker
    processes (one per core), timed from the first chunk handed out to the
    last result back; worker start-up and the copy into shared memory are
    outside the timed span.  Returns (rows per second, rows, seconds)."""
    rows = list(rows)
    handles, specs = _share({"values": values, "params": params})
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(processes=procs, initializer=_attach, initargs=(specs,)) as pool:
            pool.map(_timed_sample_chunk, [([rows[0]], seed, offset)] * procs, chunksize=1)   # warm every worker
            jobs = [(c, seed, offset) for c in _chunks(rows, procs, per_chunk=max(1, len(rows) // (2 * procs)))]
            t0 = time.perf_counter()
            done = pool.map(_timed_sample_chunk, jobs, chunksize=1)
            elapsed = time.perf_counter() - t0
    finally:
        for h in handles:
            h.close()
            h.unlink()
    n = sum(d[0] for d in done)
    return n / elapsed, n, elapsed


def _verify_tile(job):
    rows, seed, offset, row_base, extra = job
    out = verify.spec_verify(_ARRAYS["p"], _ARRAYS["q"], _ARRAYS["drafts"], seed, offset, rows=rows,
                             params=_ARRAYS["params"], row_base=row_base, **extra)
    for r in out:
        r["row_base"] = row_base
    return out


def spec_verify_tiled(p_values, q_values, drafts, seed, offset, row_bases, params=None, procs=None, **extra):
    """oracle.verify.spec_verify over every row of the batch once per entry
    of row_bases (the batch verified as parts of a larger batch that repeats
    its logits, each part with its own uniforms); one result list, tile by
    tile, each result also carrying its "row_base"."""
    procs = procs or default_procs()
    rows = list(range(np.asarray(p_values).shape[0]))
    jobs = [(rows, seed, offset, int(base), extra) for base in row_bases]
    return _run({"p": p_values, "q": q_values, "drafts": drafts, "params": params}, _verify_tile, jobs, procs)
