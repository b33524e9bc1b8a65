"""GPU parity of spec_verify against the oracle (modified rejection sampling).

Same seeded inputs on both sides; drafts from the oracle's sampler (purpose
DRAFT) so they follow the transformed draft distribution.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from parity import assert_linear_parity, assert_probs, np_

pytestmark = pytest.mark.gpu


def run(zt, zd, T=1.0, top_p=1.0, top_k=0, seed=0, offset=0, drafts=None, label="", max_near=0.05):
    if drafts is None:
        drafts = oracle.sample(zd, T, top_p, top_k, seed=seed + 7, offset=offset)["tokens"]
    drafts = np.asarray(drafts, np.int64)
    g = sv.verify(zt.cuda(), zd.cuda() if zd is not None else None, torch.from_numpy(drafts).int().cuda(),
                  T, top_p, top_k, seed, offset, debug=True)
    torch.cuda.synchronize()
    r = oracle.verify(zt, zd, drafts, T, top_p, top_k, seed, offset)
    near = assert_linear_parity(g, r, max_near_frac=max_near, label=label)
    if T > 0:
        assert_probs(g["probs"], r, label)
    return g, r, near


def test_philox_matches_oracle_on_a_million_counters():
    n = 1 << 20
    for seed, row0, pos, purpose in [(0, 0, 0, 0), (12345, 2**32 - 1000, 3, 1), (2**63 + 5, 77, 9, 2)]:
        u = np_(sv.philox_uniform(seed, row0, pos, purpose, n)).astype(np.float64)
        ref = oracle.uniform(seed, np.uint64(row0) + np.arange(n, dtype=np.uint64), pos, purpose)
        np.testing.assert_array_equal(u, ref)


def test_tiny_config_64_steps():
    """tiny: B=1, gamma=4, V=1000, f32, T=1, 64 steps (stacked, offset = step)."""
    c = workloads.CONFIGS["tiny"]
    zt, zd = workloads.config_logits("tiny", 1001, steps=64)
    run(zt, zd, c["temperature"], label="tiny")


@pytest.mark.parametrize("sigma", [0.5, 1.5])
def test_nucleus_config(sigma):
    """nucleus: B=8, gamma=4, V=32000, bf16, T=0.8, top_p=0.95 (8 steps stacked)."""
    c = workloads.CONFIGS["nucleus"]
    zt, zd = workloads.config_logits("nucleus", 1002, steps=8, sd_d=sigma)
    # near-ties: a top-p crossing mass within 1e-5 of top_p is a ~1% event per row (bf16 ties)
    g, r, near = run(zt, zd, c["temperature"], c["top_p"], 0, seed=3, label=f"nucleus s={sigma}",
                     max_near=0.1)
    assert (r["accepted"] >= 0).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,top_p,top_k", [(1.0, 1.0, 0), (0.7, 1.0, 50), (1.0, 0.9, 0),
                                           (1.0, 0.8, 200), (0.5, 0.5, 3), (1.0, 1.0, 1)])
def test_transforms_ragged_vocab(dtype, T, top_p, top_k):
    """V=40001 (odd: rows start off the 16-byte grid and end in a ragged tail).
    fp32 at top_p = 0.9 has 5 near-tie sequences of the 24 on these inputs
    (top-p crossings within 1e-5 of the target mass); the others have none."""
    zt, zd = workloads.linear_logits(24, 3, 40001, 11, dtype=dtype, sd_t=3.0, sd_d=0.8)
    run(zt, zd, T, top_p, top_k, seed=5, offset=1000, label=f"{dtype} T={T} p={top_p} k={top_k}",
        max_near=0.25)


def deep_tie_logits(B, gamma, V, T, seed, dtype):
    """Rows with 3-8 tokens near the top and every other token exactly
    16 octaves (16 T ln 2) below them: the ~40000 equal tokens hold more
    than 3% of the mass, so the nucleus of top_p = 0.97 ends inside that one
    tie group, far below the keys near the maximum."""
    g = torch.Generator().manual_seed(seed)
    zt = torch.zeros(B, gamma + 1, V)
    for b in range(B):
        for k in range(gamma + 1):
            n = int(torch.randint(3, 9, (1,), generator=g))
            idx = torch.randperm(V, generator=g)[:n]
            zt[b, k, idx] = 16 * T * float(np.log(2)) + 0.05 * torch.arange(n).float()
    zd = zt[:, :gamma].clone()
    zd[zd > 0] += 0.5 * torch.rand(int((zd > 0).sum()), generator=g)
    td = torch.float32 if dtype == "f32" else torch.bfloat16
    return zt.to(td).contiguous(), zd.to(td).contiguous()


@pytest.mark.parametrize("dtype,T,top_p,top_k", [("bf16", 1.0, 0.9, 0), ("f32", 1.0, 0.95, 100),
                                                 ("bf16", 1.0, 0.95, 100)])
def test_flat_rows_overflow_the_collected_keys(dtype, T, top_p, top_k):
    """Flat rows put more keys near the maximum than each thread collects, so
    the threshold comes from the row in global memory."""
    zt, zd = workloads.linear_logits(12, 2, 40001, 23, dtype=dtype, sd_t=0.2, sd_d=0.3)
    run(zt, zd, T, top_p, top_k, seed=8, label=f"flat {dtype} p={top_p} k={top_k}", max_near=0.05)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_crossing_far_below_the_collected_keys(dtype):
    """The nucleus ends 16 octaves below the maximum (in one tie group of
    ~40000 keys); top-k = 2000 of widely spread logits likewise lies below
    the keys near the maximum."""
    zt, zd = deep_tie_logits(10, 2, 40001, 0.5, 31, dtype)
    g, r, _ = run(zt, zd, 0.5, 0.97, 0, seed=3, label=f"deep tie {dtype}", max_near=0.05)
    assert (r["accepted"] < 2).any()
    zt, zd = workloads.linear_logits(12, 2, 40001, 29, dtype=dtype, sd_t=6.0, sd_d=0.3)
    run(zt, zd, 0.5, 1.0, 2000, seed=4, label=f"wide top-k {dtype}", max_near=0.05)


@pytest.mark.parametrize("V", [1, 2, 7, 31, 999, 4097])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_and_ragged_vocabularies(V, dtype):
    zt, zd = workloads.linear_logits(40, 2, V, 20 + V, dtype=dtype, sd_t=1.5, sd_d=0.7)
    run(zt, zd, 1.0, seed=V, label=f"V={V} {dtype}")
    run(zt, zd, 0.9, 0.9, 3, seed=V + 1, label=f"V={V} {dtype} xf")


def test_bf16_ties_and_top_k_tie_inclusive():
    """Coarse bf16 logits produce many equal values; top-k keeps every tie."""
    g = torch.Generator().manual_seed(4)
    zt = (torch.randint(-6, 7, (16, 4, 3000), generator=g).float() * 0.5).bfloat16()
    zd = (zt[:, :3].float() + 0.5 * torch.randint(-1, 2, (16, 3, 3000), generator=g).float()).bfloat16()
    run(zt, zd, 1.0, 1.0, 10, seed=9, label="ties top-k")
    run(zt, zd, 1.0, 0.6, 0, seed=10, label="ties top-p")


def test_temperature_zero_is_greedy_and_reads_no_draft():
    zt, zd = workloads.linear_logits(50, 5, 5000, 31, sd_t=1.0, sd_d=0.3)
    drafts = zd.argmax(dim=2).numpy()
    g, r, _ = run(zt, zd, 0.0, drafts=drafts, label="T=0")
    g2 = sv.verify(zt.cuda(), None, torch.from_numpy(drafts).int().cuda(), 0.0)
    np.testing.assert_array_equal(np_(g2["tokens"]), np_(g["tokens"]))
    assert (r["accepted"] > 0).any() and (r["accepted"] < 5).any()


def test_large_vocab_config_full_size():
    """large_vocab at full size: B=64, gamma=7, V=128256, f32, T=1 and T=0."""
    c = workloads.CONFIGS["large_vocab"]
    zt, zd = workloads.config_logits("large_vocab", 1003)
    run(zt, zd, 1.0, seed=1, label="large_vocab T=1", max_near=0.1)
    drafts = zd.argmax(dim=2).numpy()
    run(zt, zd, 0.0, drafts=drafts, label="large_vocab T=0")


def test_stacked_steps_equal_separate_calls():
    """One call over S*B sequences (offset 0) equals S calls with offset = step*B."""
    zt, zd = workloads.config_logits("nucleus", 77, steps=6)
    drafts = torch.from_numpy(oracle.sample(zd, 0.8, 0.95, seed=1)["tokens"]).int()
    whole = sv.verify(zt.cuda(), zd.cuda(), drafts.cuda(), 0.8, 0.95, 0, 42, 0)
    B = 8
    for s in range(6):
        sl = slice(s * B, (s + 1) * B)
        part = sv.verify(zt[sl].cuda(), zd[sl].cuda(), drafts[sl].cuda(), 0.8, 0.95, 0, 42, s * B)
        for k in ("accepted", "tokens", "next_token"):
            np.testing.assert_array_equal(np_(part[k]), np_(whole[k])[sl])


def test_repeat_calls_reuse_workspace_and_are_deterministic():
    zt, zd = workloads.linear_logits(30, 4, 20000, 5, sd_t=2.0, sd_d=1.0)
    drafts = torch.from_numpy(oracle.sample(zd, 1.0, seed=2)["tokens"]).int().cuda()
    a = sv.verify(zt.cuda(), zd.cuda(), drafts, 1.0, 0.9, 20, 3, 0)
    for _ in range(3):
        b = sv.verify(zt.cuda(), zd.cuda(), drafts, 1.0, 0.9, 20, 3, 0)
        for k in ("accepted", "tokens", "next_token", "status"):
            np.testing.assert_array_equal(np_(a[k]), np_(b[k]))


def test_bad_inputs_flag_status_and_emit_nothing():
    zt, zd = workloads.linear_logits(6, 3, 3000, 8)
    zt[1, 2, 100] = float("nan")
    zd[2, 0, 5] = float("inf")
    zt[3, 1, :] = float("-inf")          # a row of only -inf
    zt[0, 0, :1000] = float("-inf")      # -inf alone is fine
    drafts = torch.from_numpy(oracle.sample(zd.nan_to_num(posinf=0.0), 1.0, seed=1)["tokens"]).int()
    drafts[4, 1] = 3000                  # out of range
    drafts[5, 0] = -1
    run(zt, zd, 1.0, seed=4, drafts=drafts.numpy(), label="bad inputs")
    r = sv.verify(zt.cuda(), zd.cuda(), drafts.cuda(), 1.0)
    assert np_(r["status"]).tolist() == [0, 4, 4, 4, 4, 4]
    assert (np_(r["tokens"])[1:] == -1).all()
    # temperature 0 reads only the target rows
    r0 = sv.verify(zt.cuda(), None, drafts.cuda(), 0.0)
    assert np_(r0["status"]).tolist() == [0, 4, 0, 4, 4, 4]


def test_host_inputs_round_trip():
    zt, zd = workloads.linear_logits(4, 3, 5000, 12)
    drafts = torch.from_numpy(oracle.sample(zd, 1.0, seed=0)["tokens"]).int()
    h = sv.verify(zt.pin_memory(), zd.pin_memory(), drafts.pin_memory(), 1.0, 1.0, 0, 0, 0)
    d = sv.verify(zt.cuda(), zd.cuda(), drafts.cuda(), 1.0, 1.0, 0, 0, 0)
    assert h["tokens"].device.type == "cpu"
    np.testing.assert_array_equal(h["tokens"].numpy(), np_(d["tokens"]))
