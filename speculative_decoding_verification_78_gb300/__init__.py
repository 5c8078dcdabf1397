"""GB300 (sm_103a) speculative-decoding verify step.

The C library libspec_verify.so (csrc/, declared in include/spec_verify.h) holds the kernels:
batched chain verification by rejection sampling, greedy and stochastic tree verification, the
temperature softmax, the drafter-side sampler and top-k, the tree-attention mask, and chain
verification fused with its LM-head GEMMs on the tensor cores. This package is its thin Python
binding (argument marshalling only); see _binding.py.
"""

from ._binding import (  # noqa: F401
    CHECKED_LIB_PATH, EXPORTS, LIB_PATH, SPEC_BF16, SPEC_CALL_CHAIN, SPEC_CALL_PROBS, SPEC_CALL_TREE,
    SPEC_ERR_ALIGN, SPEC_ERR_DTYPE, SPEC_ERR_LAUNCH, SPEC_ERR_NONFINITE, SPEC_ERR_NULL,
    SPEC_ERR_CHECK, SPEC_ERR_PARENT, SPEC_ERR_SHAPE, SPEC_ERR_TEMP, SPEC_ERR_TOKEN, SPEC_ERR_WORKSPACE, SPEC_F32,
    SPEC_MAX_GAMMA, SPEC_MAX_NODES, SPEC_MAX_V, SPEC_LMHEAD_MAX_V, SPEC_OK, SPEC_STATIC_SCRATCH_BYTES, SpecError,
    SPEC_MAX_TOPK, check, dtype_flag, load_library, new_workspace, probs, sample,
    spec_launch_shape, spec_probs, spec_sample, spec_status_string, spec_topk, spec_tree_mask,
    spec_verify_chain, spec_verify_chain_static, spec_verify_tree, spec_verify_tree_sample,
    spec_workspace_bytes,
    spec_workspace_init, topk, tree_mask, verify_chain, verify_chain_lmhead, verify_tree,
    verify_tree_sample, spec_verify_chain_lmhead, spec_lmhead_workspace_bytes, SPEC_ERR_TIMEOUT,
    spec_last_cuda_error, spec_cuda_error_string, spec_selftest_bounded_wait)
