"""libspecverify: the target model's verification step of speculative
decoding on one GB300 (sm_103a) -- tree/chain verification attention,
full-vocabulary stochastic (chain and tree) and greedy (tree) acceptance, KV
compaction, and the fused step that runs them side by side -- as hand-written
CUDA kernels behind a C ABI (include/specverify.h), with this thin Python
binding on top.
"""
from .api import (SV_BF16, SV_ERR_BAD_INPUT, SV_ERR_CUDA, SV_ERR_INVALID_ARG, SV_ERR_TIMEOUT,
                  SV_ERR_UNSUPPORTED, SV_ERR_WORKSPACE, SV_F32, SV_OK, SV_OP_TREE_ATTENTION,
                  SV_OP_VERIFY_CHAIN, SV_OP_VERIFY_STEP_CHAIN, SV_OP_VERIFY_STEP_TREE_GREEDY,
                  SV_OP_VERIFY_TREE_GREEDY, SV_OP_VERIFY_TREE_STOCHASTIC, SpecVerifyError, lib,
                  status_string, sv_compact_kv, sv_compact_kv_paged, sv_tree_attention,
                  sv_tree_attention_paged, sv_verify_chain, sv_verify_step_chain,
                  sv_verify_step_tree_greedy, sv_verify_tree_greedy, sv_verify_tree_stochastic,
                  sv_workspace_size, workspace)

__all__ = [
    "SV_BF16", "SV_F32", "SV_OK", "SV_ERR_BAD_INPUT", "SV_ERR_CUDA", "SV_ERR_INVALID_ARG",
    "SV_ERR_TIMEOUT", "SV_ERR_UNSUPPORTED", "SV_ERR_WORKSPACE", "SV_OP_TREE_ATTENTION",
    "SV_OP_VERIFY_CHAIN", "SV_OP_VERIFY_TREE_GREEDY", "SV_OP_VERIFY_TREE_STOCHASTIC",
    "SV_OP_VERIFY_STEP_CHAIN", "SV_OP_VERIFY_STEP_TREE_GREEDY",
    "SpecVerifyError", "lib", "status_string", "sv_compact_kv", "sv_compact_kv_paged",
    "sv_tree_attention", "sv_tree_attention_paged", "sv_verify_chain", "sv_verify_tree_greedy",
    "sv_verify_tree_stochastic", "sv_verify_step_chain", "sv_verify_step_tree_greedy",
    "sv_workspace_size", "workspace",
]
