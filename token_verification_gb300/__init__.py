"""GB300-native speculative-decoding verification.

The verification step (rejection sampling, greedy and tree verification) runs
in hand-written sm_103a CUDA kernels behind the C ABI of include/spec_verify.h
(libspecverify.so); this package is its Python binding plus the seeded
synthetic workload generator.  Importing the package does not load the
library; the first call does, and fails loudly if it is not built.
"""
from .api import (REQ_BAD_DRAFT_LEN, REQ_BAD_LOGITS, REQ_BAD_TOKEN, SV_BF16, SV_F32,  # noqa: F401
                  TreeOutputs, VerifyError, VerifyOutputs, alloc_outputs, spec_verify_greedy,
                  spec_verify_sample, spec_verify_tree, tree_depth, workspace)

__all__ = ["spec_verify_sample", "spec_verify_greedy", "spec_verify_tree", "alloc_outputs",
           "VerifyOutputs", "TreeOutputs", "VerifyError", "workspace", "tree_depth"]
