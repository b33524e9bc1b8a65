"""spec_verify_noalloc, the entry point for callers that cannot allocate.

Some callers may not allocate device memory when they verify (an engine
plugin whose framework owns every device allocation, a server whose device
memory budget is fixed at start-up). spec_verify_noalloc serves them with a
fixed scratch array inside the library instead of a caller workspace. These
tests call it through the C ABI and check it against spec_verify, the entry
point with a workspace, on two calls in a row: the integer outputs must be
identical and the probabilities within the parity tolerance (1e-5 relative).
This file is collected last so that a run stopping at the first failure has
run every other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from speculative_decoding_verification_05_gb300 import SpecSampling

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 * 1024 * 1024


def _outputs(B, gamma, dev):
    return {"accepted": torch.full((B,), -7, dtype=torch.int32, device=dev),
            "tokens": torch.full((B, gamma + 1), -7, dtype=torch.int32, device=dev),
            "next_token": torch.full((B,), -7, dtype=torch.int32, device=dev),
            "status": torch.full((B,), -7, dtype=torch.int32, device=dev),
            "probs": torch.full((B, gamma, 2), -7.0, dtype=torch.float32, device=dev)}


def _noalloc(lib, zt, zd, drafts, T, top_p, top_k, seed, offset, out=None):
    B, G1, V = zt.shape
    gamma = G1 - 1
    dev = zt.device
    if out is None:
        out = _outputs(B, gamma, dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)
    dt = sv.SPEC_F32 if zt.dtype == torch.float32 else sv.SPEC_BF16
    stream = torch.cuda.current_stream(dev)
    rc = lib.spec_verify_noalloc(p(zt), p(zd), dt, p(drafts), B, gamma, V,
                                 SpecSampling(T, top_p, top_k), seed, offset,
                                 p(out["accepted"]), p(out["tokens"]), p(out["next_token"]),
                                 p(out["status"]), p(out["probs"]), ctypes.c_void_p(stream.cuda_stream))
    assert rc == sv.SPEC_OK, lib.spec_status_string(rc)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype,V,T,top_p,top_k", [("bf16", 32000, 0.8, 0.95, 0), ("f32", 40001, 1.0, 1.0, 0),
                                                   ("f32", 5000, 0.0, 1.0, 0)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dtype, V, T, top_p, top_k):
    lib = sv.load_library()
    zt, zd = workloads.linear_logits(16, 4, V, 321, dtype=dtype, sd_t=3.0, sd_d=0.8)
    drafts = oracle.sample(zd, T, top_p, top_k, seed=6)["tokens"]
    zt, zd = zt.cuda(), zd.cuda()
    d = torch.from_numpy(drafts).int().cuda()
    ref = sv.verify(zt, zd, d, T, top_p, top_k, 11, 5, debug=True)
    torch.cuda.synchronize()
    for _ in range(2):
        got = _noalloc(lib, zt, zd if T > 0 else None, d, T, top_p, top_k, 11, 5)
        for k in ("accepted", "tokens", "next_token", "status"):
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=k)
        np.testing.assert_allclose(got["probs"].cpu().numpy(), ref["probs"].cpu().numpy(), rtol=1e-5, atol=0)


def test_noalloc_takes_no_device_memory_after_its_first_call():
    """The first call on a device may load the scratch array's module (and
    commit its memory); every later call must leave the device's free memory
    unchanged. Outputs are allocated before the calls, so nothing else
    allocates in between."""
    lib = sv.load_library()
    zt, zd = workloads.linear_logits(8, 4, 32000, 77, dtype="bf16", sd_t=3.0, sd_d=0.8)
    drafts = torch.from_numpy(oracle.sample(zd, 0.8, 0.95, 0, seed=3)["tokens"]).int().cuda()
    zt, zd = zt.cuda(), zd.cuda()
    out = _outputs(8, 4, zt.device)
    _noalloc(lib, zt, zd, drafts, 0.8, 0.95, 0, 1, 0, out)
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(lib, zt, zd, drafts, 0.8, 0.95, 0, 1, 0, out)
        assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = sv.load_library()
    need = lambda B: lib.spec_verify_workspace_size(B, 4, 32000, sv.SPEC_BF16)
    B = 1
    while need(B) <= SCRATCH_BYTES:
        B *= 2
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.spec_verify_noalloc(fake, fake, sv.SPEC_BF16, fake, B, 4, 32000, SpecSampling(1.0, 1.0, 0),
                                 0, 0, fake, fake, fake, None, None, None)
    assert rc == sv.SPEC_EINVAL
