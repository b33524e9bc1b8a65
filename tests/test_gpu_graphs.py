"""The C-ABI calls inside a CUDA graph: they only enqueue a memset and
kernels on the caller's stream (no allocation, no synchronisation), so a
serving loop can capture a verification step once and replay it. Replays give
the same outputs as eager calls on the same inputs.
"""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_05_gb300 as sv
import workloads
from parity import np_

pytestmark = pytest.mark.gpu


def test_verify_and_tree_steps_replay_from_a_graph():
    c = workloads.CONFIGS["nucleus"]
    zt, zd = workloads.config_logits("nucleus", 41, steps=1, device="cuda")
    drafts = workloads.gumbel_drafts(zd, c["temperature"], 2)
    z, tok, par, dep = workloads.tree_inputs(16, 64, 32016, 41, device="cpu")
    z, tok, par, dep = z.cuda(), tok.cuda(), par.cuda(), dep.cuda()
    cand = torch.from_numpy(workloads.rest_candidates(16, 256, 16, 32016, 41)).cuda()
    root = torch.zeros(16, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        # eager calls first: they also size the cached workspaces
        want = sv.verify(zt, zd, drafts, c["temperature"], c["top_p"], 0, 5, 0)
        want_t = sv.verify_tree(z, tok, par, dep, 6)
        want_b = sv.tree_build(cand, root, 32016, 64)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            got = sv.verify(zt, zd, drafts, c["temperature"], c["top_p"], 0, 5, 0)
            got_t = sv.verify_tree(z, tok, par, dep, 6)
            got_b = sv.tree_build(cand, root, 32016, 64)
        for _ in range(3):
            g.replay()
        stream.synchronize()
    for k in ("accepted", "tokens", "next_token", "status"):
        np.testing.assert_array_equal(np_(got[k]), np_(want[k]), err_msg=k)
    for k in ("accept_len", "path_nodes", "tokens", "bonus", "status"):
        np.testing.assert_array_equal(np_(got_t[k]), np_(want_t[k]), err_msg=k)
    for k in ("node_tokens", "parent", "depth", "mask", "n_nodes"):
        np.testing.assert_array_equal(np_(got_b[k]), np_(want_b[k]), err_msg=k)
