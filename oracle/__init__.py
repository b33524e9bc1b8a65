"""CPU oracle for speculative-decoding verification (test infrastructure).

This package is TEST INFRASTRUCTURE. It is a plain, slow, fp64 restatement of
what the verification step computes, written from the pages that define the
method. Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
leg of ``bench.py`` (and ``bench.py --impl reference``) may import it. The
product path (the CUDA library and its Python binding) never imports, calls or
links anything here, and nothing here imports the product path.

Sources (cited by page title and section throughout):

* [SpS]    "Accelerating Large Language Model Decoding with Speculative
           Sampling" (reading notes on Chen et al., 2023): sections
           "改进的拒绝采样" (modified rejection sampling: acceptance probability,
           resampling from (q-p)+, bonus token), "与标准采样方法的兼容性"
           (temperature / top-k / nucleus applied before the scheme), and the
           appendix proof of Theorem 1.
* [SD]     "Fast Inference from Transformers via Speculative Decoding"
           (write-up of Leviathan et al., ICML 2023): "方法细节" (acceptance
           rule, standardised sampling, E[#tokens], alpha, walltime and
           operation factors), appendix E worked example.
* [REST]   "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法"
           (REST, retrieval-based speculative decoding): section
           "REST: 基于检索的投机解码" (trie with prefix counts, the heaviest
           subtree, BFS pseudo-sequence and tree attention mask, exact-match
           acceptance).
* [Mentor] "推测解码的一种最优有损变体" (an optimal lossy variant of
           speculative decoding): sections "导师解码" and "解决优化问题".

Notation follows [SpS] and [Mentor]: q is the target distribution, p the draft.

Parity status per function (see the pins in ``tests/test_oracle_*.py``):
every function is pinned except the exact numeric value of the mentor alpha
for a given (q, p, D), which the pages pin only through properties
(feasibility, monotonicity, optimality on a grid, D=0 and KL(q||p)<=D limits);
that part is "parity unpinned" beyond those properties.
"""

from .philox import philox4x32_10, uniform, PURPOSE_ACCEPT, PURPOSE_RESAMPLE, PURPOSE_DRAFT, PURPOSE_NOISE
from .spec import (
    NEAR_TIE,
    STATUS_OK,
    STATUS_EDATA,
    transformed_probs,
    accept_test,
    inverse_cdf,
    verify,
    verify_tree,
    verify_mentor,
    mentor_solve,
    mentor_pi,
    sample,
    acceptance_rate,
    expected_tokens,
    walltime_factor,
    ops_factor,
    best_gamma,
    estimate_alpha,
)
from .rest import MAX_COUNT as REST_MAX_COUNT, rest_tree, rest_tree_batch
