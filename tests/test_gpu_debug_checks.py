"""The debug build of the library, with device-side index checks.

libspecverify_debug.so is built from the same sources with -DSPEC_DEBUG: the
kernels check the indices they compute (every global write, the workspace,
token and shared-memory indexing) against the extent of the array each
addresses; a failed check skips the access, is counted (spec_debug_failures)
and marks the sequence's status SPEC_EBOUNDS, so nothing traps. This stands
in for a memory checker, which cannot be run here. Every entry point runs
through it on vocabularies from 3 to 64 and on a few larger shapes (the
shared-memory row path, long rows split into segments): no check may fail,
the linear verifications must match the oracle, and the other entry points
must return what the release build returns.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from parity import assert_linear_parity, np_

pytestmark = pytest.mark.gpu


def _failures():
    lib = sv.load_library(sv.DEBUG_LIB_PATH)
    line = ctypes.c_int(0)
    n = lib.spec_debug_failures(ctypes.byref(line))
    return n, line.value


@pytest.fixture(scope="module")
def dbg():
    lib = sv.load_library(sv.DEBUG_LIB_PATH)
    assert lib.spec_debug_build() == 1 and sv.load_library().spec_debug_build() == 0
    assert _failures() == (0, 0)
    yield lib
    assert _failures() == (0, 0)


def _both(fn):
    """fn() through the release and the debug library."""
    rel = fn()
    with sv.use_library(sv.DEBUG_LIB_PATH):
        deb = fn()
    torch.cuda.synchronize()
    n, line = _failures()
    assert n == 0, f"{n} index checks failed, the first at line {line}"
    return rel, deb


def _same(rel, deb, keys):
    for k in keys:
        np.testing.assert_array_equal(np_(deb[k]), np_(rel[k]), err_msg=k)


@pytest.mark.parametrize("V", [3, 5, 8, 16, 31, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_small_vocabularies(dbg, V, dtype):
    zt, zd = workloads.linear_logits(9, 3, V, 100 + V, dtype=dtype, sd_t=1.5, sd_d=0.7)
    for T, top_p, top_k in [(1.0, 1.0, 0), (0.8, 0.9, 2), (0.0, 1.0, 0)]:
        drafts = oracle.sample(zd, T, top_p, top_k, seed=V)["tokens"]
        d = torch.from_numpy(drafts).int().cuda()
        rel, deb = _both(lambda: sv.verify(zt.cuda(), zd.cuda() if T > 0 else None, d, T, top_p, top_k, 3, 0))
        _same(rel, deb, ("accepted", "tokens", "next_token", "status"))
        r = oracle.verify(zt, zd, drafts, T, top_p, top_k, 3, 0)
        assert_linear_parity(deb, r, max_near_frac=0.0, label=f"debug V={V} {dtype} T={T}")


def test_verify_shared_memory_rows_and_segments(dbg):
    zt, zd = workloads.linear_logits(6, 4, 32000, 7, dtype="bf16", sd_t=3.0, sd_d=0.5, boost=6.0, boost_p=0.01)
    drafts = torch.from_numpy(oracle.sample(zd, 0.8, 0.95, 0, seed=1)["tokens"]).int().cuda()
    rel, deb = _both(lambda: sv.verify(zt.cuda(), zd.cuda(), drafts, 0.8, 0.95, 0, 1, 0))
    _same(rel, deb, ("accepted", "tokens", "next_token", "status"))
    zt, zd = workloads.linear_logits(2, 3, 50000, 8, sd_t=2.0, sd_d=0.5)   # few long rows: segments
    drafts = torch.from_numpy(oracle.sample(zd, 1.0, seed=2)["tokens"]).int().cuda()
    rel, deb = _both(lambda: sv.verify(zt.cuda(), zd.cuda(), drafts, 1.0, 1.0, 0, 2, 0))
    _same(rel, deb, ("accepted", "tokens", "next_token", "status"))


@pytest.mark.parametrize("V", [3, 64, 5000])
def test_other_entry_points(dbg, V):
    zt, zd = workloads.linear_logits(5, 3, V, 50 + V, sd_t=2.0, sd_d=1.2)
    drafts = torch.from_numpy(oracle.sample(zd, 1.0, seed=5)["tokens"]).int().cuda()
    rel, deb = _both(lambda: sv.verify_mentor(zt.cuda(), zd.cuda(), drafts, 1.0, 0.05, 30, 4, 0))
    _same(rel, deb, ("accepted", "tokens", "next_token", "status", "alpha", "beta"))
    rel, deb = _both(lambda: sv.sample(zt.cuda(), 0.9, 0.9, 0, seed=1, offset=0))
    _same(rel, deb, ("tokens", "status"))
    rel, deb = _both(lambda: sv.acceptance_rate(zt.cuda(), zd.cuda(), 1.0, 0.9, 0))
    _same(rel, deb, ("beta", "status"))
    z, tok, par, dep = workloads.tree_inputs(3, 16, max(V, 64), 9)  # distinct sibling tokens need V >= 4
    rel, deb = _both(lambda: sv.verify_tree(z.cuda(), tok.cuda(), par.cuda(), dep.cuda(), 6))
    _same(rel, deb, ("accept_len", "path_nodes", "tokens", "bonus", "status"))
    cand = workloads.rest_candidates(3, 20, 6, max(V, 8), 6)
    root = torch.tensor([1, 2, 0], dtype=torch.int32)
    rel, deb = _both(lambda: sv.tree_build(torch.from_numpy(cand).cuda(), root.cuda(), max(V, 8), 16))
    _same(rel, deb, ("node_tokens", "parent", "depth", "mask", "n_nodes", "status"))


def test_a_withheld_copy_times_out_and_the_device_stays_usable(dbg):
    """The first CTA of the shared-memory row kernel withholds the copy of its
    second row: nothing completes that buffer's barrier, the CTA's bounded
    waits give up, the rows it had left (rows 1 x grid, 2 x grid, ...) are
    reported as timed out, every other sequence is verified as the release
    library verifies it, and the next call (copy no longer withheld) is
    complete and correct."""
    B, G, V = 60, 4, 32000
    zt, zd = workloads.linear_logits(B, G, V, 77, dtype="bf16", sd_t=3.0, sd_d=0.5, boost=6.0, boost_p=0.01)
    drafts = torch.from_numpy(oracle.sample(zd, 0.8, 0.95, 0, seed=3)["tokens"]).int().cuda()
    zt, zd = zt.cuda(), zd.cuda()
    rel = sv.verify(zt, zd, drafts, 0.8, 0.95, 0, 4, 0)
    rows, R = B * (2 * G + 1), 2 * G + 1
    grid = min(rows, torch.cuda.get_device_properties(0).multi_processor_count)
    lost = sorted({r // R for r in range(grid, rows, grid)})
    assert lost, "the first CTA must take more than one row"
    assert dbg.spec_debug_withhold_copy(1) == 0
    try:
        with sv.use_library(sv.DEBUG_LIB_PATH):
            got = sv.verify(zt, zd, drafts, 0.8, 0.95, 0, 4, 0)
        torch.cuda.synchronize()
    finally:
        assert dbg.spec_debug_withhold_copy(-1) == 0
    st = np_(got["status"])
    assert (st[lost] == 3).all(), st[lost]  # SPEC_ETIMEOUT
    assert (np_(got["accepted"])[lost] == -1).all()
    keep = np.setdiff1d(np.arange(B), lost)
    assert (st[keep] == 0).all()
    for k in ("accepted", "tokens", "next_token"):
        np.testing.assert_array_equal(np_(got[k])[keep], np_(rel[k])[keep], err_msg=k)
    rel2, deb2 = _both(lambda: sv.verify(zt, zd, drafts, 0.8, 0.95, 0, 4, 0))
    _same(rel2, deb2, ("accepted", "tokens", "next_token", "status"))
    assert (np_(deb2["status"]) == 0).all()
