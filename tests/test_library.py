"""The C-ABI library: it builds, loads, exports every symbol the header
declares, and rejects invalid arguments on the host (no GPU needed: an invalid
call returns SPEC_EINVAL before any CUDA call)."""

import ctypes
import os
import re

import pytest

import speculative_decoding_verification_05_gb300 as sv
from speculative_decoding_verification_05_gb300 import SpecSampling

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")
EINVAL = 1


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sv.LIB_PATH):
        from speculative_decoding_verification_05_gb300 import build
        build.build()
    return sv.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = _declared()
    assert "spec_verify" in names and "spec_verify_tree" in names and "spec_verify_mentor" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(sv.EXPORTED) == sorted(n for n in names)


def test_version_and_status_strings(lib):
    assert lib.spec_version() == 100
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(4) == b"SPEC_EDATA"
    assert lib.spec_last_cuda_error() == b""


def test_workspace_sizes_are_positive_and_grow(lib):
    a = lib.spec_verify_workspace_size(8, 4, 32000, 1)
    b = lib.spec_verify_workspace_size(64, 7, 128256, 0)
    assert 0 < a and 0 < b and a % 256 == 0 and b % 256 == 0
    assert lib.spec_verify_workspace_size(16, 4, 32000, 1) > a
    # bf16 shapes the shared-memory row path can take also hold the kept list
    # of every target row (1024 entries of a 4-byte index and a 2-byte logit)
    assert a - lib.spec_verify_workspace_size(8, 4, 32000, 0) >= 8 * 5 * 1024 * 6
    assert lib.spec_verify_workspace_size(8, 4, 32001, 1) == lib.spec_verify_workspace_size(8, 4, 32001, 0)
    assert lib.spec_verify_workspace_size(0, 4, 10, 0) == 0
    assert lib.spec_verify_tree_workspace_size(16, 64, 32016, 0) > 0
    m = lib.spec_verify_mentor_workspace_size(32, 5, 32128, 0)
    assert m > lib.spec_verify_workspace_size(32, 5, 32128, 0)
    assert lib.spec_sample_workspace_size(4, 3, 100, 0) > 0


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below is invalid


def _verify(lib, **kw):
    a = dict(target=FAKE, draft=FAKE, dtype=0, toks=FAKE, B=2, gamma=3, V=100,
             samp=SpecSampling(1.0, 1.0, 0), ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.spec_verify(a["target"], a["draft"], a["dtype"], a["toks"], a["B"], a["gamma"], a["V"],
                           a["samp"], 0, 0, FAKE, FAKE, FAKE, None, None, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw", [
    dict(B=0), dict(gamma=0), dict(gamma=256), dict(V=0), dict(V=262145), dict(dtype=7),
    dict(target=None), dict(toks=None), dict(ws=None), dict(ws_bytes=16),
    dict(draft=None), dict(samp=SpecSampling(-1.0, 1.0, 0)), dict(samp=SpecSampling(1.0, 0.0, 0)),
    dict(samp=SpecSampling(1.0, 1.5, 0)), dict(samp=SpecSampling(1.0, float("nan"), 0)),
    dict(samp=SpecSampling(float("inf"), 1.0, 0)), dict(samp=SpecSampling(1.0, 1.0, -2)),
    dict(target=ctypes.c_void_p((1 << 20) + 2)), dict(ws=ctypes.c_void_p((1 << 20) + 16)),
])
def test_verify_rejects_bad_arguments(lib, kw):
    assert _verify(lib, **kw) == EINVAL


def test_tree_mentor_sample_reject_bad_arguments(lib):
    T = lambda **k: lib.spec_verify_tree(k.get("t", FAKE), 0, FAKE, FAKE, FAKE, k.get("B", 2), k.get("N", 8),
                                         k.get("V", 100), k.get("md", 3), FAKE, FAKE, FAKE, FAKE, None,
                                         FAKE, 1 << 30, None)
    assert T(N=0) == EINVAL and T(N=1025) == EINVAL and T(md=8) == EINVAL and T(md=-1) == EINVAL
    assert T(t=None) == EINVAL
    M = lambda **k: lib.spec_verify_mentor(FAKE, FAKE, 0, FAKE, 2, 3, 100, k.get("T", 1.0), k.get("D", 0.1),
                                           k.get("it", 30), 0, 0, FAKE, FAKE, FAKE, None, None, None, None,
                                           FAKE, k.get("ws", 1 << 34), None)
    assert M(T=0.0) == EINVAL and M(D=-0.1) == EINVAL and M(it=0) == EINVAL and M(it=65) == EINVAL
    assert M(D=float("nan")) == EINVAL and M(ws=64) == EINVAL
    S = lambda **k: lib.spec_sample(FAKE, 0, k.get("B", 2), k.get("P", 1), 100, k.get("s", SpecSampling(1, 1, 0)),
                                    0, 0, 0, 2, FAKE, None, FAKE, 1 << 30, None)
    assert S(B=0) == EINVAL and S(P=0) == EINVAL and S(s=SpecSampling(1, 2, 0)) == EINVAL


@pytest.mark.parametrize("l", [0.0, -0.5, 1.5, float("nan"), float("inf")])
def test_lenient_verify_rejects_bad_lenience(lib, l):
    rc = lib.spec_verify_lenient(FAKE, FAKE, 0, FAKE, 2, 3, 100, SpecSampling(1.0, 1.0, 0), l, 0, 0,
                                 FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None)
    assert rc == EINVAL


def test_tree_build_rejects_bad_arguments(lib):
    def T(**k):
        a = dict(cand=FAKE, B=2, C=8, L=4, V=100, N=16, tok=FAKE, nn=FAKE)
        a.update(k)
        return lib.spec_tree_build(a["cand"], None, FAKE, a["B"], a["C"], a["L"], a["V"], a["N"],
                                   a["tok"], FAKE, FAKE, None, a["nn"], None, None)
    for kw in (dict(B=0), dict(C=0), dict(C=1025), dict(L=0), dict(L=33), dict(C=512, L=16),
               dict(V=0), dict(N=1), dict(N=1025), dict(cand=None), dict(tok=None), dict(nn=None),
               dict(cand=ctypes.c_void_p((1 << 20) + 2))):
        assert T(**kw) == EINVAL, kw


def test_planner_matches_oracle(lib):
    import math

    import numpy as np

    import oracle
    rng = np.random.default_rng(4)
    for _ in range(300):
        a = float(rng.choice([0.0, 1.0, rng.random()]))
        g = int(rng.integers(0, 40))
        c = float(rng.choice([0.0, rng.random(), 10 * rng.random()]))
        assert sv.expected_tokens(a, g) == pytest.approx(oracle.expected_tokens(a, g), rel=1e-14)
        assert sv.walltime_factor(a, g, c) == pytest.approx(oracle.walltime_factor(a, g, c), rel=1e-14)
        assert sv.ops_factor(a, g, c) == pytest.approx(oracle.ops_factor(a, g, c), rel=1e-14)
        if g >= 1 and a < 0.999:
            assert sv.best_gamma(a, c, g) == oracle.best_gamma(a, c, g)
    # the appendix E worked example: zero-cost draft, alpha 0.9, gamma 10
    assert round(sv.walltime_factor(0.9, 10, 0.0), 2) == 6.86 and round(sv.ops_factor(0.9, 10, 0.0), 1) == 1.6
    for bad in ((-0.1, 3), (1.1, 3), (float("nan"), 3), (0.5, -1)):
        assert math.isnan(sv.expected_tokens(*bad))
    assert math.isnan(sv.walltime_factor(0.5, 3, -1.0)) and math.isnan(sv.ops_factor(0.5, 3, float("inf")))
    assert sv.best_gamma(0.5, 0.1, 0) == -1 and sv.best_gamma(2.0, 0.1, 5) == -1 and sv.best_gamma(0.5, -1, 5) == -1


def test_acceptance_rate_rejects_bad_arguments(lib):
    def A(**k):
        a = dict(t=FAKE, d=FAKE, B=2, G=3, V=100, s=SpecSampling(1.0, 1.0, 0), beta=FAKE, ws=FAKE)
        a.update(k)
        return lib.spec_acceptance_rate(a["t"], a["d"], 0, a["B"], a["G"], a["V"], a["s"], a["beta"], None,
                                        a["ws"], 1 << 30, None)
    for kw in (dict(B=0), dict(G=0), dict(V=0), dict(t=None), dict(d=None), dict(beta=None), dict(ws=None),
               dict(s=SpecSampling(0.0, 1.0, 0)), dict(s=SpecSampling(1.0, 0.0, 0)),
               dict(beta=ctypes.c_void_p((1 << 20) + 2))):
        assert A(**kw) == EINVAL, kw
