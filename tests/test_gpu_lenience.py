"""GPU parity of spec_verify_lenient against the oracle's lenient verification
(acceptance min(1, q/(l p)), residual max(0, q - l p)); l = 1 must equal
spec_verify bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from parity import assert_linear_parity, assert_probs, np_

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("l", [0.1, 0.5, 0.9])
@pytest.mark.parametrize("name,T,top_p,top_k", [("tiny", 1.0, 1.0, 0), ("nucleus", 0.8, 0.95, 0),
                                                ("mentor", 1.0, 0.9, 20)])
def test_lenient_matches_oracle(l, name, T, top_p, top_k):
    zt, zd = workloads.config_logits(name, 41, steps=4)
    drafts = oracle.sample(zd, T, top_p, top_k, seed=3)["tokens"]
    g = sv.verify(zt.cuda(), zd.cuda(), torch.from_numpy(drafts).int().cuda(), T, top_p, top_k, 9, 2,
                  debug=True, lenience=l)
    torch.cuda.synchronize()
    r = oracle.verify(zt, zd, drafts, T, top_p, top_k, 9, 2, lenience=l)
    assert_linear_parity(g, r, max_near_frac=0.05, label=f"{name} l={l}")
    assert_probs(g["probs"], r, f"{name} l={l}")
    if l <= 0.5:
        # leniency accepts more than the exact method on the same uniforms
        e = oracle.verify(zt, zd, drafts, T, top_p, top_k, 9, 2)
        assert r["accepted"].mean() > e["accepted"].mean()


def test_lenience_one_equals_spec_verify():
    """spec_verify_lenient with l = 1, called through the C ABI, equals spec_verify."""
    import ctypes
    zt, zd = workloads.config_logits("nucleus", 43, steps=2)
    d = torch.from_numpy(oracle.sample(zd, 0.8, 0.95, 0, seed=4)["tokens"]).int().cuda()
    zt, zd = zt.cuda(), zd.cuda()
    a = sv.verify(zt, zd, d, 0.8, 0.95, 0, 5, 0, debug=True)
    lib = sv.load_library()
    B, G1, V = zt.shape
    o = {k: torch.full_like(v, -7) for k, v in a.items()}
    ws = torch.empty(lib.spec_verify_workspace_size(B, G1 - 1, V, sv.SPEC_BF16), dtype=torch.uint8, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.spec_verify_lenient(P(zt), P(zd), sv.SPEC_BF16, P(d), B, G1 - 1, V, sv.SpecSampling(0.8, 0.95, 0),
                                 1.0, 5, 0, P(o["accepted"]), P(o["tokens"]), P(o["next_token"]), P(o["status"]),
                                 P(o["probs"]), P(ws), ws.numel(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == sv.SPEC_OK
    torch.cuda.synchronize()
    for k in ("accepted", "tokens", "next_token", "status", "probs"):
        np.testing.assert_array_equal(np_(o[k]), np_(a[k]), err_msg=k)
