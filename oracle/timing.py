"""Times the oracle on every host core: the CPU baseline that bench.py reports.

TEST INFRASTRUCTURE (see the package docstring). Nothing here computes any
part of the method. It calls the oracle's own functions, unchanged, on a
bounded sample of a workload: once in the calling process (one core), and in
one worker process per host core, all running at the same time. Workers are
started with the 'spawn' method, which is safe next to a CUDA context (a
process forked after the first CUDA call can hang), and each is held to one
thread of numerical libraries.
"""

import multiprocessing as mp
import os
import time

from . import rest, spec

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def host_cores():
    """Cores this process may run on (its affinity mask)."""
    if hasattr(os, "sched_getaffinity"):
        return len(os.sched_getaffinity(0))
    return os.cpu_count() or 1


def run_once(job, n):
    """One oracle call on the job's sample (n varies the seed and the Philox
    row offset, as consecutive steps would). Returns the positions verified."""
    k = job["kind"]
    if k == "verify":
        B, G = job["drafts"].shape
        spec.verify(job["zt"], job["zd"] if job["T"] > 0 else None, job["drafts"], job["T"], job["top_p"], 0,
                    seed=n, offset=n * B, lenience=job.get("lenience", 1.0))
        return B * G
    if k == "mentor":
        B, G = job["drafts"].shape
        spec.verify_mentor(job["zt"], job["zd"], job["drafts"], job["T"], job["kl_bound"], job["iters"],
                           seed=n, offset=n * B)
        return B * G
    if k == "tree":
        z = job["z"]
        spec.verify_tree(z, job["tok"], job["par"], job["dep"], job["max_depth"])
        return z.shape[0] * (z.shape[1] - 1)
    if k == "rest":
        t = rest.rest_tree_batch(job["cand"], None, job["root"], job["N"], job["V"])
        spec.verify_tree(job["z"], t["tokens"], t["parent"], t["depth"], job["max_depth"])
        return job["cand"].shape[0] * (job["N"] - 1)
    if k == "alpha":
        zt, zd = job["zt"], job["zd"]
        B, G1, V = zt.shape
        q, _ = spec.transformed_probs(zt[:, :G1 - 1].reshape(-1, V), job["T"], 0, job["top_p"])
        p, _ = spec.transformed_probs(zd.reshape(-1, V), job["T"], 0, job["top_p"])
        spec.acceptance_rate(q, p)
        return B * (G1 - 1)
    raise ValueError(f"unknown job kind {k}")


def time_one_core(job, budget_s):
    """Positions per second of the oracle in this process; (rate, calls, seconds)."""
    t0 = time.perf_counter()
    n = pos = 0
    while True:
        pos += run_once(job, n)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            return pos / dt, n, dt


def _worker(job, budget_s, rounds, barrier, out_q, wid):
    for rnd in range(rounds):
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        n = pos = 0
        while True:
            pos += run_once(job, 1000003 * wid + 1009 * rnd + n)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        out_q.put((rnd, wid, n, pos, dt))


def time_all_cores(job, budget_s, rounds=1, workers=None):
    """Aggregate positions per second of `workers` (default: every host core)
    concurrent oracle processes, for each of `rounds` rounds of `budget_s`
    seconds that all workers start together. Returns (rates, workers, calls),
    rates[r] the sum over workers of their positions / seconds in round r."""
    workers = workers or host_cores()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(workers)
    out_q = ctx.Queue()
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    for v in _THREAD_VARS:
        os.environ[v] = "1"
    try:
        procs = [ctx.Process(target=_worker, args=(job, budget_s, rounds, barrier, out_q, i), daemon=True)
                 for i in range(workers)]
        for p in procs:
            p.start()
    finally:
        for v, x in saved.items():
            if x is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = x
    res = [out_q.get(timeout=600 + 2 * budget_s * rounds) for _ in range(workers * rounds)]
    for p in procs:
        p.join(timeout=60)
    rates = [0.0] * rounds
    calls = 0
    for rnd, _, n, pos, dt in res:
        rates[rnd] += pos / dt
        calls += n
    return rates, workers, calls
