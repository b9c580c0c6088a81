"""Batched draft-token verification for speculative decoding on GB300 (sm_103a).

The work runs in libspecverify.so (hand-written CUDA behind the C ABI of
include/spec_verify.h); this package is the torch-facing binding:

    spec_verify_stochastic  acceptance u <= min(1, p/q), first rejection, residual or
                            bonus token by inverse CDF, with NKL and the greedy decision
    spec_verify_greedy      argmax-match verification
    spec_verify_tree        longest accepted root-to-leaf path of a draft tree
    spec_nkl                KL(q || p) / ln V per position
"""
from .api import (Workspace, spec_nkl, spec_tree_depth, spec_verify_greedy, spec_verify_stochastic,
                  spec_verify_tree, spec_workspace_bytes)

__all__ = ["Workspace", "spec_nkl", "spec_tree_depth", "spec_verify_greedy", "spec_verify_stochastic",
           "spec_verify_tree", "spec_workspace_bytes"]
