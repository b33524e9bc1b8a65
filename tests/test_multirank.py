"""The multi-rank path of bench.py, on CPU with gloo (world size 2).

Verification shards by sequence with no exchange: rank r verifies global
sequences [r B, (r + 1) B) with Philox row base r B, so the ranks' results
put together are the single-device results of the whole batch (checked here
with the oracle standing in for each rank's device work). The job's time is
the slowest rank's; under torchrun the reference arm runs on rank 0 only and
prints one line.
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    zt, zd = workloads.config_logits("tiny", 31, steps=8)      # 8 sequences
    B = zt.shape[0] // world
    sl = slice(rank * B, (rank + 1) * B)
    off = bench.shard_offset(rank, B)
    drafts = oracle.sample(zd[sl], 1.0, seed=5, offset=off)["tokens"]
    r = oracle.verify(zt[sl], zd[sl], drafts, 1.0, 0.9, 0, 9, off)
    ms = bench.max_over_ranks(10.0 + rank, torch.device("cpu"))
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), drafts=drafts, accepted=r["accepted"], tokens=r["tokens"],
             next_token=r["next_token"], ms=ms)
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_ranks_equal_one_device(tmp_path):
    mp.spawn(_rank, args=(WORLD, _free_port(), str(tmp_path)), nprocs=WORLD, join=True)
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(WORLD)]
    zt, zd = workloads.config_logits("tiny", 31, steps=8)
    drafts = oracle.sample(zd, 1.0, seed=5, offset=0)["tokens"]
    whole = oracle.verify(zt, zd, drafts, 1.0, 0.9, 0, 9, 0)
    np.testing.assert_array_equal(np.concatenate([p["drafts"] for p in parts]), drafts)
    for k in ("accepted", "tokens", "next_token"):
        np.testing.assert_array_equal(np.concatenate([p[k] for p in parts]), whole[k])
    # every rank reports the slowest rank's time
    assert [float(p["ms"]) for p in parts] == [11.0, 11.0]
    # whole-job throughput: all ranks' positions over that time
    assert bench.job_value(WORLD, 32, 10, 11.0) == WORLD * 32 * 10 / 0.011


def test_reference_arm_prints_once_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={WORLD}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", str(WORLD), "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-budget", "0.3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == WORLD and d["value"] > 0
