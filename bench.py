"""Throughput benchmark of the verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One bench step is one pass of the whole verification path over one batch. The
default workload is the large-vocabulary configuration (B=64, gamma=7,
V=128256, f32 logits, temperature 1): 20 of its 200 steps are stacked into
one call over 1280 sequences (offset = step * B, so every Philox counter is
the one a step-by-step loop would use), 9.85 GB of logits resident in HBM,
larger than L2, so no flush is needed between timed steps. Workloads smaller
than twice L2 (tiny) overwrite a 256 MB buffer before each timed step,
outside the timed events. ``--stack S`` overrides the number of stacked
steps (a smaller case of the same workload, used for ncu captures).

The same run also times the other V >= 32k workloads (nucleus x1000 steps,
large-vocab at temperature 0, the tree workload, the mentor workload) and
reports each under ``per_workload`` with its own roofline and clocks
(``--no-extra`` skips them).

Prints one JSON line: verified positions/s (whole job), the roofline of the
timed call (algorithmic bytes / CUDA-event time against the measured HBM copy
bandwidth), the CPU oracle baseline (one core and every host core), the
end-to-end figure through the public API with host buffers, launch count and
SM clocks during the run. Under torchrun (N > 1) every rank runs an
independent replica (the path shards by sequence with no exchange), and rank 0
reports the aggregate.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verified positions/sec and achieved HBM GB/s vs GB300 roofline (1 GPU)"
UNIT = "positions/s"

WORKLOADS = {
    # name: (config, steps stacked into one call, temperature override)
    "large_vocab": ("large_vocab", 20, 1.0),
    "large_vocab_t0": ("large_vocab", 20, 0.0),
    "nucleus": ("nucleus", 1000, None),
    "tree": ("tree", 32, None),
    "mentor": ("mentor", 250, None),
    "tiny": ("tiny", 64, None),
    "rest": ("rest", 4, None),
    "nucleus_lenient": ("nucleus", 1000, None),
    "nucleus_alpha": ("nucleus", 1000, None),
}
DEFAULT = "large_vocab"
# the other V >= 32k workloads, timed in the same run as the default one
EXTRA = ("nucleus", "large_vocab_t0", "tree", "mentor")
LENIENCE = {"nucleus_lenient": 0.5}   # lenient verification (l < 1); others are exact
OPS = {"nucleus_alpha": "alpha"}      # measured acceptance probabilities instead of verification

# The timed unit is one library call; where a call launches several kernels the
# label names them all (the row or argmax kernel reads every logit byte).
SMEM_PATH = "smem_row_kernel + smem_tail_kernel + smem_fulldraw_kernel"
KERNEL_OF = {"nucleus": SMEM_PATH, "tiny": "row_kernel<f32> + draw_kernel",
             "large_vocab": "row_kernel<f32> + draw_kernel", "large_vocab_t0": "argmax_kernel<f32>",
             "tree": "argmax_kernel<f32>",
             "mentor": "row_kernel<f32> + mentor_kernel + mentor_resolve_kernel",
             "nucleus_lenient": SMEM_PATH,
             "rest": "tree_build_kernel + argmax_kernel<f32>",
             "nucleus_alpha": "row_kernel<bf16,transform> (records) + beta_kernel"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def shard_offset(rank, batch):
    """Philox row base of a rank's sequences: rank r verifies global sequences
    [r * batch, (r + 1) * batch), so every random number is the one a single
    device verifying the whole job would draw for that sequence."""
    return rank * batch


def max_over_ranks(ms, device):
    """The slowest rank's time (the job is as fast as its slowest replica)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, positions_per_step, steps, total_ms):
    """Whole-job throughput: every rank's positions over the slowest rank's time."""
    return world * positions_per_step * steps / (total_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_sources_sha():
    """Hash of the library's CUDA sources: a recorded ncu traffic figure holds
    only for the kernels it was taken on."""
    import hashlib

    h = hashlib.sha256()
    src = os.path.join(ROOT, "speculative_decoding_verification_05_gb300", "csrc")
    for f in sorted(os.listdir(src)):
        with open(os.path.join(src, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, stacked):
    """Per-launch DRAM bytes (read + write) of the timed call from the committed
    ncu summary, or None: none recorded, another stacking, or kernels changed
    since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if e is None or e.get("stacked") != stacked or e.get("csrc_sha16") != kernel_sources_sha():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def make_inputs(name, steps_stacked, temperature, device, seed=2024, lenience=1.0, rank=0):
    """Synthetic inputs of a workload on the device (generator: workloads.py)."""
    import speculative_decoding_verification_05_gb300 as sv

    c = dict(workloads.CONFIGS[name])
    if c["kind"] == "rest":
        B = c["B"] * steps_stacked
        cand = torch.from_numpy(workloads.rest_candidates(B, c["C"], c["L"], c["V"], seed, bases=c["bases"],
                                                          diverge=c["diverge"])).to(device)
        root = torch.from_numpy(np.random.default_rng(seed).integers(0, c["V"], B).astype(np.int32)).to(device)
        t = sv.tree_build(cand, root, c["V"], c["N"], with_mask=False)   # the tree, to force its logits
        z = workloads.forced_tree_logits(t["node_tokens"].cpu().numpy(), t["parent"].cpu().numpy(),
                                         t["n_nodes"].cpu().numpy(), c["V"], seed, sd=c["sd"],
                                         force_p=c["force_p"], device=device)
        return dict(kind="rest", cand=cand, root=root, z=z, B=B, N=c["N"], V=c["V"], C=c["C"], L=c["L"],
                    max_depth=c["L"], esize=4)
    if c["kind"] == "tree":
        B = c["B"] * steps_stacked
        z, tok, par, dep = workloads.tree_inputs(B, c["N"], c["V"], seed, device="cpu")
        return dict(kind="tree", z=z.to(device), tok=tok.to(device), par=par.to(device), dep=dep.to(device),
                    B=B, N=c["N"], V=c["V"], max_depth=c["max_depth"], esize=4)
    T = c["temperature"] if temperature is None else temperature
    zt, zd = workloads.config_logits(name, seed, steps=steps_stacked, device=device)
    B = zt.shape[0]
    top_p = c.get("top_p", 1.0)
    # drafts: the library's own sampler on the transformed draft distribution
    offset = shard_offset(rank, B)
    drafts = sv.sample(zd, T, top_p, 0, seed=seed, offset=offset, purpose=sv.PURPOSE_DRAFT)["tokens"]
    return dict(kind=c["kind"], zt=zt, zd=zd, drafts=drafts, B=B, gamma=c["gamma"], V=c["V"], T=T, lenience=lenience,
                offset=offset,
                top_p=top_p, kl_bound=c.get("kl_bound", 0.0), iters=c.get("iters", 30),
                esize=zt.element_size())


def run_step(inp):
    import speculative_decoding_verification_05_gb300 as sv

    if inp.get("op") == "alpha":
        return sv.acceptance_rate(inp["zt"], inp["zd"], inp["T"], inp["top_p"], 0)
    if inp["kind"] == "rest":
        t = sv.tree_build(inp["cand"], inp["root"], inp["V"], inp["N"])
        return sv.verify_tree(inp["z"], t["node_tokens"], t["parent"], t["depth"], inp["max_depth"])
    if inp["kind"] == "tree":
        return sv.verify_tree(inp["z"], inp["tok"], inp["par"], inp["dep"], inp["max_depth"])
    if inp["kind"] == "mentor":
        return sv.verify_mentor(inp["zt"], inp["zd"], inp["drafts"], inp["T"], inp["kl_bound"], inp["iters"],
                                0, inp["offset"])
    return sv.verify(inp["zt"], inp["zd"], inp["drafts"], inp["T"], inp["top_p"], 0, 0, inp["offset"],
                     lenience=inp["lenience"])


def run_step_host(inp, host):
    """End-to-end through the public API: pinned host inputs in, host outputs back."""
    import speculative_decoding_verification_05_gb300 as sv

    if inp.get("op") == "alpha":
        return sv.acceptance_rate(host["zt"], host["zd"], inp["T"], inp["top_p"], 0)
    if inp["kind"] == "rest":
        # two public calls on host buffers: the tree (and its mask) comes back in between
        t = sv.tree_build(host["cand"], host["root"], inp["V"], inp["N"])
        r = sv.verify_tree(host["z"], t["node_tokens"], t["parent"], t["depth"], inp["max_depth"])
        return {**{"tree_" + k: v for k, v in t.items()}, **r}
    if inp["kind"] == "tree":
        return sv.verify_tree(host["z"], host["tok"], host["par"], host["dep"], inp["max_depth"])
    if inp["kind"] == "mentor":
        return sv.verify_mentor(host["zt"], host["zd"], host["drafts"], inp["T"], inp["kl_bound"], inp["iters"],
                                0, inp["offset"])
    return sv.verify(host["zt"], host["zd"], host["drafts"], inp["T"], inp["top_p"], 0, 0, inp["offset"],
                     lenience=inp["lenience"])


def algorithmic(inp):
    """(bytes, verified positions) one step must read / decides."""
    if inp.get("op") == "alpha":
        # each of the 2 gamma rows of a position pair read once (the bonus row is not needed)
        B, G = inp["B"], inp["gamma"]
        return B * 2 * G * inp["V"] * inp["esize"], B * G
    if inp["kind"] == "rest":
        # logits once, the candidates once, the tree arrays and mask written once
        B, N = inp["B"], inp["N"]
        extra = B * inp["C"] * inp["L"] * 4 + B * N * (3 * 4 + N) + B * 2 * 4
        return (workloads.algorithmic_bytes("rest", B, inp["V"], 4, N=N) + extra,
                workloads.verified_positions("rest", B, N=N))
    if inp["kind"] == "tree":
        return (workloads.algorithmic_bytes("tree", inp["B"], inp["V"], inp["esize"], N=inp["N"]),
                workloads.verified_positions("tree", inp["B"], N=inp["N"]))
    return (workloads.algorithmic_bytes("linear", inp["B"], inp["V"], inp["esize"], gamma=inp["gamma"],
                                        temperature=inp["T"]),
            workloads.verified_positions("linear", inp["B"], gamma=inp["gamma"]))


def smem_path(inp):
    """Whether spec_verify takes the shared-memory row path for these inputs:
    bf16 logits with a top-k / top-p transform, V a multiple of 8 and at
    most about 54000 (a ring of two rows fits), both tensors on 16 bytes."""
    zt, zd = inp.get("zt"), inp.get("zd")
    return (inp["kind"] == "linear" and inp.get("op", "verify") == "verify" and inp["T"] > 0
            and inp["esize"] == 2 and inp["top_p"] < 1.0 and inp["V"] % 8 == 0 and inp["V"] <= 54000
            and zt is not None and zd is not None and zt.data_ptr() % 16 == 0 and zd.data_ptr() % 16 == 0)


def launches_per_step(inp):
    """Kernels one library call launches: rows, position solve and resolve
    (mentor); the argmax kernel (tree, T = 0); on the shared-memory row path
    the row kernel, the fallback-and-draw kernel and the full-row draw
    kernel; rows and draws otherwise."""
    if inp["kind"] == "mentor":
        return 3
    if inp["kind"] == "rest" or inp.get("op") == "alpha":
        return 2
    if inp["kind"] == "tree" or inp["T"] == 0:
        return 1
    if smem_path(inp):
        return 3
    return 2


def oracle_job(name, temperature, lenience=1.0, op="verify", seed=99):
    """A bounded sample of the workload for the oracle: one step of the
    configuration (two of its 64 sequences for the large vocabulary, whose
    rows are 4x longer), as numpy arrays."""
    import oracle

    c = dict(workloads.CONFIGS[name])
    if op == "alpha":
        zt, zd = workloads.config_logits(name, seed, steps=1)
        return dict(kind="alpha", zt=zt.float().numpy(), zd=zd.float().numpy(), T=c["temperature"],
                    top_p=c.get("top_p", 1.0)), f"beta of one step (B={c['B']}, V={c['V']})"
    if c["kind"] == "rest":
        B = c["B"]
        cand = workloads.rest_candidates(B, c["C"], c["L"], c["V"], seed, bases=c["bases"], diverge=c["diverge"])
        root = np.arange(B, dtype=np.int32)
        tr = oracle.rest_tree_batch(cand, None, root, c["N"], c["V"])
        z = workloads.forced_tree_logits(tr["tokens"], tr["parent"], tr["n_nodes"], c["V"], seed, sd=c["sd"],
                                         force_p=c["force_p"])
        return (dict(kind="rest", cand=cand, root=root, z=z.numpy() if hasattr(z, "numpy") else z, N=c["N"],
                     V=c["V"], max_depth=c["L"]),
                f"one REST step: {B} trees built (C={c['C']}, L={c['L']}, N={c['N']}) and verified (V={c['V']})")
    if c["kind"] == "tree":
        z, tok, par, dep = workloads.tree_inputs(c["B"], c["N"], c["V"], seed)
        return (dict(kind="tree", z=z.numpy(), tok=tok.numpy(), par=par.numpy(), dep=dep.numpy(),
                     max_depth=c["max_depth"]), f"one step: {c['B']} trees (N={c['N']}, V={c['V']})")
    T = c.get("temperature", 0.0) if temperature is None else temperature
    B = 2 if name == "large_vocab" else c["B"]
    zt, zd = workloads.linear_logits(B, c["gamma"], c["V"], seed, dtype=c["dtype"], sd_t=c["sd_t"],
                                     sd_d=c["sd_d"], boost=c.get("boost", 0.0), boost_p=c.get("boost_p", 0.0),
                                     zipf=c.get("zipf", 0.0))
    top_p = c.get("top_p", 1.0)
    drafts = oracle.sample(zd, T, top_p, 0, seed=seed)["tokens"]
    job = dict(kind="mentor" if c["kind"] == "mentor" else "verify", zt=zt.float().numpy(), zd=zd.float().numpy(),
               drafts=drafts, T=T, top_p=top_p, lenience=lenience, kl_bound=c.get("kl_bound", 0.0),
               iters=c.get("iters", 30))
    return job, f"{B} sequences of one step (gamma={c['gamma']}, V={c['V']}, T={T})"


def cpu_baseline(name, temperature, budget_s=6.0, lenience=1.0, op="verify"):
    """The oracle, as it stands, on a bounded sample of the workload: one host
    core, then every host core at once (one spawned process per core)."""
    from oracle import timing

    job, what = oracle_job(name, temperature, lenience, op)
    one, n1, dt1 = timing.time_one_core(job, budget_s)
    rates, cores, calls = timing.time_all_cores(job, budget_s)
    return {"value": rates[0], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{what}; {calls} oracle calls over {cores} concurrent processes in {budget_s:.0f} s",
            "single_core": {"value": one, "cores": 1, "sample": f"{n1} oracle calls in {dt1:.1f} s"}}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import timing

    cfg, _, temp = WORKLOADS[args.workload]
    lv = LENIENCE.get(args.workload, 1.0)
    budget = args.ref_budget if args.ref_budget > 0 else max(1.5, 60.0 / max(1, args.steps + args.warmup))
    job, what = oracle_job(cfg, temp, lv, OPS.get(args.workload, "verify"))
    rates, cores, calls = timing.time_all_cores(job, budget, rounds=args.warmup + args.steps)
    timed = rates[args.warmup:]
    v = statistics.median(timed)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(args.workload, WORKLOADS[args.workload][1])},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{what}; each step {budget:.1f} s on {cores} concurrent processes "
                                       f"(median of {args.steps} steps after {args.warmup} warm-up)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def describe(name, stacked):
    """The workload as the JSON line names it: configuration, sizes, stacking."""
    cfg, _, temp = WORKLOADS[name]
    c = workloads.CONFIGS[cfg]
    T = c.get("temperature") if temp is None else temp
    desc = {"large_vocab": f"B={c['B']}, gamma={c.get('gamma')}, V={c['V']}, f32, T={T}",
            "nucleus": f"B={c['B']}, gamma={c.get('gamma')}, V={c['V']}, bf16, T={T}, top_p={c.get('top_p')}",
            "tree": f"B={c['B']}, N={c.get('N')}, V={c['V']}, f32",
            "mentor": f"B={c['B']}, gamma={c.get('gamma')}, V={c['V']}, f32, T=1, D={c.get('kl_bound')}, "
                      f"{c.get('iters')} bisection steps"}.get(cfg, f"B={c['B']}, V={c['V']}")
    extra = f", lenience {LENIENCE[name]}" if name in LENIENCE else ""
    extra += ", acceptance rates (beta) only" if name in OPS else ""
    return f"{name}: {cfg} ({desc}{extra}), {stacked} steps stacked in one call of B={c['B'] * stacked} sequences"


def measure(args, name, stacked, steps, warmup, device, ws, rank, local):
    """Times `steps` calls of one workload (after `warmup`); returns its figures."""
    cfg, _, temp = WORKLOADS[name]
    inp = make_inputs(cfg, stacked, temp, device, seed=2024 + rank, lenience=LENIENCE.get(name, 1.0), rank=rank)
    inp["op"] = OPS.get(name, "verify")
    nbytes, npos = algorithmic(inp)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(device)

    l2_bytes = 129 * 2**20
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=device) if nbytes < 2 * l2_bytes else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    # clocks are sampled from the warm-up through the timed steps; a short
    # timed region is followed by untimed steps until 0.3 s of load is sampled
    with ClockSampler(local) as clk:
        t_load0 = time.perf_counter()
        for _ in range(warmup):
            if flush is not None:
                flush.fill_(1)
            run_step(inp)
        barrier()
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 255)  # evicts the previous step's inputs from L2 (untimed)
            starts[i].record(stream)
            run_step(inp)
            ends[i].record(stream)
        barrier()
        while time.perf_counter() - t_load0 < 0.3:
            run_step(inp)
            torch.cuda.synchronize(device)
    per_launch_ms = [st.elapsed_time(en) for st, en in zip(starts, ends)]
    total_ms = max_over_ranks(sum(per_launch_ms), device)
    # acceptance statistics of one step (a property of the synthetic inputs)
    out = run_step(inp)
    torch.cuda.synchronize(device)
    acc_mean = None
    if "accepted" in out:
        acc_mean = float(out["accepted"].float().mean().item())
    elif "accept_len" in out:
        acc_mean = float(out["accept_len"].float().mean().item())
    alpha_est = float(out["beta"].float().mean().item()) if inp.get("op") == "alpha" else None
    peak, peak_kind = measured_peaks()
    avg_launch_ms = statistics.mean(per_launch_ms)
    achieved = nbytes / (avg_launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic(name, stacked), "kernel": KERNEL_OF[name],
            "algorithmic_bytes_per_launch": nbytes, "peak_source": f"{peak_kind} hbm_gbs (copy)",
            "frac_of_nominal_8TBps": achieved / 8000.0}
    return dict(inp=inp, nbytes=nbytes, npos=npos, total_ms=total_ms, ms_per_step=total_ms / steps,
                value=job_value(ws, npos, steps, total_ms), roofline=roof,
                clocks=dict(clk.summary(), window="warm-up + timed steps (+ untimed steps up to 0.3 s)"),
                mean_accepted=acc_mean, alpha=alpha_est, cfg=cfg, stacked=stacked, flush=flush is not None,
                batch=inp["B"], launches=launches_per_step(inp),
                workload=describe(name, stacked))


def e2e_figure(inp, steps, device, ws, npos):
    """The same metric through the public API with pinned host buffers: the
    inputs' host-to-device copies and the outputs' device-to-host copies are
    inside the timed region."""
    host = {k: v.to("cpu").pin_memory() for k, v in inp.items() if isinstance(v, torch.Tensor)}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    for _ in range(2):
        run_step_host(inp, host)
    torch.cuda.synchronize(device)
    n_e2e = max(3, min(steps, 10))
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        r = run_step_host(inp, host)
    dt = max_over_ranks((time.perf_counter() - t0) * 1e3, device) / 1e3
    d2h = sum(v.numel() * v.element_size() for v in r.values() if isinstance(v, torch.Tensor))
    return {"value": ws * npos * n_e2e / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "ms_per_step": dt * 1e3 / n_e2e,
            "h2d_gbs": h2d / (dt / n_e2e) / 1e9}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other V >= 32k workloads")
    ap.add_argument("--stack", type=int, default=0, help="stacked steps per call (default: the workload's)")
    ap.add_argument("--ref-budget", type=float, default=0.0,
                    help="reference arm: seconds of oracle work per step (default: about 60 s over all steps)")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    assert args.warmup >= 3, "at least 3 warm-up steps"

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    import speculative_decoding_verification_05_gb300 as sv

    sv.load_library()
    stacked = args.stack if args.stack > 0 else WORKLOADS[args.workload][1]
    m = measure(args, args.workload, stacked, args.steps, args.warmup, device, ws, rank, local)
    inp = m["inp"]
    e2e = None if args.no_e2e else e2e_figure(inp, args.steps, device, ws, m["npos"])
    del inp, m["inp"]
    extra = {}
    if not args.no_extra and args.workload == DEFAULT and args.stack == 0:
        for name in EXTRA:
            torch.cuda.empty_cache()
            x = measure(args, name, WORKLOADS[name][1], max(3, min(args.steps, 10)), 3, device, ws, rank, local)
            del x["inp"]
            extra[name] = {"workload": x["workload"], "value": x["value"], "unit": UNIT,
                           "ms_per_step": x["ms_per_step"], "steps": max(3, min(args.steps, 10)),
                           "roofline": x["roofline"], "clocks": x["clocks"], "mean_accepted": x["mean_accepted"],
                           "bytes_per_step": x["nbytes"], "positions_per_step": x["npos"]}
    if rank != 0:
        return 0
    cfg = m["cfg"]
    cpu = None if args.no_cpu else cpu_baseline(cfg, WORKLOADS[args.workload][2],
                                                lenience=LENIENCE.get(args.workload, 1.0),
                                                op=OPS.get(args.workload, "verify"))
    esize = workloads.TORCH_DTYPE[workloads.CONFIGS[cfg].get("dtype", "f32")].itemsize
    line = {
        "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if esize == 2 else "f32", "data": "synthetic",
        "config": {"workload": m["workload"], "global_batch": m["batch"] * ws,
                   "bytes_per_step": m["nbytes"], "positions_per_step": m["npos"],
                   "l2": "L2 flushed between steps" if m["flush"] else "inputs larger than 2x L2 (no flush)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": m["roofline"], "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": m["launches"] * args.steps,
        "clocks": m["clocks"], "hbm_gbs": m["roofline"]["achieved"], "mean_accepted": m["mean_accepted"],
        **({"alpha": m["alpha"]} if m["alpha"] is not None else {}),
        **({"per_workload": extra} if extra else {}),
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
