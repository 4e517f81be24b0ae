// sv_api.cu -- the extern "C" boundary of libspecverify: argument checks on
// the host (nothing is launched when they fail), then the kernel launches.
// Declarations and the contract of every call are in include/specverify.h.
#include <cmath>
#include <cstdint>

#include "sv_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(sv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

int sv_version(void) { return 100; }  // 0.1.0

const char *sv_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "SV_OK";
        case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: invalid argument";
        case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing or too small";
        case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: shape outside the supported range";
        case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA runtime call failed";
        case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded wait in a kernel gave up";
        case SV_ERR_BAD_INPUT: return "SV_ERR_BAD_INPUT: invalid per-sequence input";
    }
    return "unknown sv_status";
}

size_t sv_workspace_size(sv_op op, int B, int T_or_N, int V, sv_dtype dtype, int Hq, int Hkv,
                         int D) {
    if (B <= 0 || T_or_N <= 0) return 0;
    switch (op) {
        case SV_OP_TREE_ATTENTION: {
            if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
            sv::AttnPlan pl;
            // (the workspace does not depend on the cache length)
            if (sv::plan_attention(B, T_or_N, Hq, Hkv, D, 1 << 30, &pl) != SV_OK) return 0;
            return pl.bytes;
        }
        case SV_OP_VERIFY_CHAIN:
        case SV_OP_VERIFY_TREE_GREEDY: {
            if (V <= 0 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
            // the shapes the calls refuse as unsupported have no size
            if (T_or_N > (op == SV_OP_VERIFY_CHAIN ? 63 : 1024) || V >= (1 << 30)) return 0;
            const sv::VocabPlan pl = sv::plan_vocab(op == SV_OP_VERIFY_CHAIN, B, T_or_N, V, dtype);
            if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return 0;
            return pl.bytes;
        }
        case SV_OP_VERIFY_TREE_STOCHASTIC: {
            if (V <= 0 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
            if (T_or_N > 1024 || V > (1 << 22)) return 0;
            const sv::VocabPlan pl = sv::plan_vocab_stree(B, T_or_N, V, dtype);
            if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return 0;
            return pl.bytes;
        }
        case SV_OP_VERIFY_STEP_CHAIN:
        case SV_OP_VERIFY_STEP_TREE_GREEDY: {
            const bool chain = op == SV_OP_VERIFY_STEP_CHAIN;
            if (V <= 0 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
            if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
            if (T_or_N > (chain ? 63 : 1024) || V >= (1 << 30) || (!chain && Hkv > 256)) return 0;
            const sv::VocabPlan pl = sv::plan_vocab(chain, B, T_or_N, V, dtype);
            if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return 0;
            return sv::step_workspace_size(chain, B, T_or_N, V, dtype, Hq, Hkv, D);
        }
    }
    return 0;
}

sv_status sv_tree_attention(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *prefix_lens, const int32_t *parents,
                            const int32_t *node_counts, int B, int T, int Hq, int Hkv, int D,
                            int S_max, float scale, void *out, int32_t *seq_status,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    if (!q || !k_cache || !v_cache || !prefix_lens || !out) return SV_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || S_max < T) return SV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !(scale > 0.f) || !std::isfinite(scale)) return SV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return SV_ERR_INVALID_ARG;
    if ((long long)B * Hkv * S_max >= (1LL << 31)) return SV_ERR_UNSUPPORTED;
    sv::AttnPlan pl;
    const sv_status st = sv::plan_attention(B, T, Hq, Hkv, D, S_max, &pl);
    if (st != SV_OK) return st;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    sv::AttnArgs a{q,   k_cache, v_cache, prefix_lens, parents,    B,       T, Hq, Hkv, D,
                   S_max, scale, out,  seq_status, nullptr, 0, 0, 0, node_counts};
    return sv::launch_tree_attention(a, pl, workspace, as_stream(stream));
}

static bool valid_page_size(int ps) {
    // a power of two from 8 (one swizzle atom of rows) up, or a multiple of the 128-key tile
    return ps >= 8 && ((ps & (ps - 1)) == 0 || ps % 128 == 0);
}

sv_status sv_tree_attention_paged(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *block_table, int max_pages, int num_pages,
                                  int page_size, const int32_t *prefix_lens,
                                  const int32_t *parents, const int32_t *node_counts, int B,
                                  int T, int Hq, int Hkv, int D, float scale, void *out,
                                  int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                  sv_stream_t stream) {
    if (!q || !k_pages || !v_pages || !block_table || !prefix_lens || !out) return SV_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_pages <= 0 || num_pages <= 0)
        return SV_ERR_INVALID_ARG;
    if (!valid_page_size(page_size)) return SV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !(scale > 0.f) || !std::isfinite(scale)) return SV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
        return SV_ERR_INVALID_ARG;
    const long long S_max = (long long)max_pages * page_size;
    if (S_max < T) return SV_ERR_INVALID_ARG;
    if ((long long)num_pages * Hkv * page_size >= (1LL << 31) || S_max >= (1LL << 30))
        return SV_ERR_UNSUPPORTED;
    sv::AttnPlan pl;
    const sv_status st = sv::plan_attention(B, T, Hq, Hkv, D, (int)S_max, &pl);
    if (st != SV_OK) return st;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    sv::AttnArgs a{q,  k_pages, v_pages, prefix_lens, parents,     B,         T,        Hq,
                   Hkv, D,      (int)S_max, scale,     out,         seq_status, block_table,
                   max_pages, num_pages, page_size, node_counts};
    return sv::launch_tree_attention(a, pl, workspace, as_stream(stream));
}

sv_status sv_verify_chain(const void *target_logits, const void *draft_logits, sv_dtype dtype,
                          const int32_t *draft_tokens, const int32_t *draft_lens,
                          const float *u_accept, const float *u_sample, int B, int N, int V,
                          int32_t *accepted_len, int32_t *out_tokens, float *probs_out,
                          int32_t *seq_status, void *workspace, size_t workspace_bytes,
                          sv_stream_t stream) {
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample ||
        !accepted_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || V <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SV_ERR_INVALID_ARG;
    if (N > 63 || V >= (1 << 30)) return SV_ERR_UNSUPPORTED;
    const sv::VocabPlan pl = sv::plan_vocab(true, B, N, V, dtype);
    if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return SV_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    sv::ChainArgs a{target_logits, draft_logits, draft_tokens, draft_lens, u_accept, u_sample,
                    B,             N,            V,            accepted_len, out_tokens,
                    probs_out,     seq_status};
    return sv::launch_verify_chain(a, dtype, pl, workspace, as_stream(stream));
}

sv_status sv_verify_tree_greedy(const void *target_logits, sv_dtype dtype,
                                const int32_t *node_tokens, const int32_t *parents,
                                const int32_t *node_counts, int B, int T, int V,
                                int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                                int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                sv_stream_t stream) {
    if (!target_logits || !node_tokens || !accepted_len || !path_nodes || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || V <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(target_logits)) return SV_ERR_INVALID_ARG;
    if (T > 1024 || V >= (1 << 30)) return SV_ERR_UNSUPPORTED;
    const sv::VocabPlan pl = sv::plan_vocab(false, B, T, V, dtype);
    if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return SV_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    sv::TreeArgs a{target_logits, node_tokens, parents,    node_counts, B, T, V, accepted_len,
                   path_nodes,    out_tokens,  seq_status};
    return sv::launch_verify_tree_greedy(a, dtype, pl, workspace, as_stream(stream));
}

sv_status sv_verify_tree_stochastic(const void *target_logits, const void *draft_logits,
                                    sv_dtype dtype, const int32_t *node_tokens,
                                    const int32_t *parents, const int32_t *node_counts,
                                    const float *u_accept, const float *u_sample, int B, int T,
                                    int V,
                                    int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                                    int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                    sv_stream_t stream) {
    if (!target_logits || !draft_logits || !node_tokens || !u_accept || !u_sample ||
        !accepted_len || !path_nodes || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || V <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SV_ERR_INVALID_ARG;
    if (T > 1024 || V > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const sv::VocabPlan pl = sv::plan_vocab_stree(B, T, V, dtype);
    if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return SV_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    sv::STreeArgs a{target_logits, draft_logits, node_tokens, parents,    node_counts, u_accept,
                    u_sample,      B,            T,           V,          accepted_len, path_nodes,
                    out_tokens,    seq_status};
    return sv::launch_verify_tree_stochastic(a, dtype, pl, workspace, as_stream(stream));
}

sv_status sv_compact_kv(void *k_cache, void *v_cache, const int32_t *prefix_lens,
                        int32_t *new_kv_lens, const int32_t *path_nodes, int path_stride,
                        const int32_t *accepted_len, int B, int Hkv, int D, int S_max,
                        int32_t *seq_status, sv_stream_t stream) {
    if (!k_cache || !v_cache || !prefix_lens || !new_kv_lens || !accepted_len)
        return SV_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || D <= 0 || S_max <= 0) return SV_ERR_INVALID_ARG;
    if (path_nodes && path_stride <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return SV_ERR_INVALID_ARG;
    if (D % 8 != 0 || D > 256) return SV_ERR_UNSUPPORTED;
    sv::CompactArgs a{k_cache, v_cache, prefix_lens, new_kv_lens, path_nodes, path_stride,
                      accepted_len, B, Hkv, D, S_max, seq_status, nullptr, 0, 0};
    return sv::launch_compact_kv(a, as_stream(stream));
}

sv_status sv_compact_kv_paged(void *k_pages, void *v_pages, const int32_t *block_table,
                              int max_pages, int num_pages, int page_size,
                              const int32_t *prefix_lens, int32_t *new_kv_lens,
                              const int32_t *path_nodes, int path_stride,
                              const int32_t *accepted_len, int B, int Hkv, int D,
                              int32_t *seq_status, sv_stream_t stream) {
    if (!k_pages || !v_pages || !block_table || !prefix_lens || !new_kv_lens || !accepted_len)
        return SV_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || D <= 0 || max_pages <= 0 || num_pages <= 0 || page_size <= 0)
        return SV_ERR_INVALID_ARG;
    if (path_nodes && path_stride <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(k_pages) || !aligned16(v_pages)) return SV_ERR_INVALID_ARG;
    if (D % 8 != 0 || D > 256) return SV_ERR_UNSUPPORTED;
    const long long S_max = (long long)max_pages * page_size;
    if (S_max >= (1LL << 30) || (long long)num_pages * Hkv * page_size >= (1LL << 31))
        return SV_ERR_UNSUPPORTED;
    sv::CompactArgs a{k_pages, v_pages,    prefix_lens, new_kv_lens, path_nodes, path_stride,
                      accepted_len, B, Hkv, D, (int)S_max, seq_status, block_table, max_pages,
                      page_size};
    a.num_pages = num_pages;
    return sv::launch_compact_kv(a, as_stream(stream));
}

}  // extern "C"
