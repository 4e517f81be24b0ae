// sv_internal.h -- host-side plans and launchers shared between the C ABI
// (sv_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/specverify.h"

namespace sv {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch `fn` with programmatic stream serialisation: the grid may begin
// launching once the stream's previous kernel lets it (or ends), overlapping
// that kernel's tail.  Every kernel of this library starts with
// griddep_wait(), so it reads nothing before its predecessor has finished.
inline cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, void **args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---------------------------------------------------------------- vocabulary pass

// Per (row, chunk) statistics written by the streaming pass.
struct RowPartial {
    float m;     // max of logit * log2(e) over the chunk
    float s;     // sum of exp2(logit * log2(e) - m)
    float best;  // largest logit (argmax mode)
    int idx;     // its index, smallest among equal maxima; INT_MAX if none
};

// Per-sequence result of the chain decisions, taken at the start of the residual draw.
struct ChainDecision {
    int a;       // first rejected position, N_b if all accepted, -1 if the sequence is invalid
    int n_draft; // N_b, the sequence's draft length
    float ms_t;  // target row a: max * log2(e) and normaliser
    float s_t;
    float ms_d;  // draft row a (unused when a == N)
    float s_d;
    float pad2[2];
};

struct VocabPlan {
    int rows_per_seq;     // 2N+1 (chain) or T (tree)
    int nchunks;          // streaming chunks per row
    int chunk_elems;
    int res_chunks;       // residual-draw chunks per sequence (chain only)
    int res_chunk_elems;
    int walk_cluster;     // CTAs per sequence of the stochastic tree walk (set at launch)
    int max_ctas;         // cap on the streaming pass's persistent grid (0: one CTA per SM)
    bool vec;             // rows are 16-byte aligned: vector loads
    int recs_per_unit;    // chain: (max, sum) records per (row, chunk)
    size_t off_counters;  // 2*B + 4 ints: arrivals per sequence, then [2*B] a timeout flag
    size_t off_partials;  // B * rows_per_seq * nchunks RowPartial
    size_t off_chunktot;  // B * res_chunks float2
    size_t bytes;
};

VocabPlan plan_vocab(bool chain, int B, int rows_or_n, int V, int dtype);

constexpr int kMaxResChunks = 256;  // chunks of a row in the chain's residual draw, at most
constexpr int kMaxResCluster = 16;  // chunks of a row for the residual draw's cluster form, at most

struct ChainArgs {
    const void *target;
    const void *draft;
    const int32_t *tokens;
    const int32_t *draft_lens;  // per-sequence N_b (0 <= N_b <= N), or null: all N
    const float *u_accept;
    const float *u_sample;
    int B, N, V;
    int32_t *accepted_len;
    int32_t *out_tokens;
    float *probs;
    int32_t *seq_status;
    // fused step only (null otherwise): new_kv_lens[b] = prefix_lens[b] + a + 1
    // when the sequence's cache holds its nodes (prefix_lens[b] + N_b + 1 <= S_max), else prefix_lens[b]
    const int32_t *prefix_lens;
    int32_t *new_kv_lens;
    int S_max;
};

// Compaction folded into a fused tree step: the K/V rows of (sequence b, KV
// head h) move once both the attention has finished reading them and the
// path is known.  step_ctr[b * Hkv + h] counts those arrivals (rg_count row
// groups of the attention, then the walk); whoever brings it to
// rg_count + 1 moves the rows and resets it.
// The walk's side of the hook holds a head's moved rows in registers, room for
// T - 1 = 63 accepted rows: the attention's node limit (T <= 64).
constexpr int kStepHookMaxT = 64;

struct StepHook {
    int *step_ctr;             // [B * Hkv], zero between calls
    uint4 *k, *v;              // contiguous caches [B, Hkv, S_max, D] as 16-byte words
    const int32_t *prefix_lens;
    int32_t *new_kv_lens;      // written by the walk
    int Hkv, rg_count, S_max, D;
};

struct TreeArgs {
    const void *target;
    const int32_t *tokens;
    const int32_t *parents;
    const int32_t *node_counts;  // per-sequence T_b (1 <= T_b <= T), or null: all T
    int B, T, V;
    int32_t *accepted_len;
    int32_t *path_nodes;
    int32_t *out_tokens;
    int32_t *seq_status;
    // fused step only: the compaction hook (step_ctr null otherwise), and
    // new_kv_lens / prefix_lens written without it when the step compacts in
    // a kernel of its own (then step_ctr null and new_kv_lens null)
    StepHook hook;
};

// Stochastic (multi-draft) acceptance on a tree.
struct STreeArgs {
    const void *target;  // [B, T, V]
    const void *draft;   // [B, T, V]: row u is the distribution u's children were drawn from
    const int32_t *tokens;
    const int32_t *parents;      // or null: a chain
    const int32_t *node_counts;  // per-sequence T_b (1 <= T_b <= T), or null: all T
    const float *u_accept;       // [B, T]
    const float *u_sample;   // [B]
    int B, T, V;
    int32_t *accepted_len;
    int32_t *path_nodes;
    int32_t *out_tokens;
    int32_t *seq_status;
};

// Workspace of the stochastic tree walk: (max, sum) per (sequence, row, chunk).
VocabPlan plan_vocab_stree(int B, int T, int V, int dtype);
sv_status launch_verify_tree_stochastic(const STreeArgs &args, int dtype, const VocabPlan &plan,
                                        void *ws, cudaStream_t stream);

sv_status launch_verify_chain(const ChainArgs &args, int dtype, const VocabPlan &plan, void *ws,
                              cudaStream_t stream);
sv_status launch_verify_tree_greedy(const TreeArgs &args, int dtype, const VocabPlan &plan,
                                    void *ws, cudaStream_t stream);

// ---------------------------------------------------------------- attention

struct AttnPlan {
    int stages;       // K/V pipeline depth
    int mrows;        // the MMA's M: 64 or 128
    int rows_per_rg;  // query rows per row group: the largest multiple of G <= mrows
    int rg;           // row groups per (sequence, KV head)
    int grid;         // CTAs launched
    int cluster;      // CTAs per cluster in cluster mode (one cluster per row group), else 1
    int smem;         // dynamic shared memory bytes
    size_t off_pair_ctr;
    size_t off_part_o;
    size_t off_part_ml;
    size_t bytes;
};

// max_ctas > 0 caps the CTAs the call may use (a fused step leaves the
// rest of the SMs to the vocabulary pass); 0: the whole device.
sv_status plan_attention(int B, int T, int Hq, int Hkv, int D, int S_max, AttnPlan *plan,
                         int max_ctas = 0);

// tcgen05 attention kernel (sv_attention_tc.cu)
struct AttnKParams;
int tc_smem_bytes(int stages, int mrows, int B);
const void *tc_kernel_fn(int stages, int mrows);

struct AttnArgs {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *prefix_lens;
    const int32_t *parents;
    int B, T, Hq, Hkv, D, S_max;  // S_max = max_pages * page_size for a paged cache
    float scale;
    void *out;
    int32_t *seq_status;
    const int32_t *block_table;  // null: contiguous caches [B, Hkv, S_max, D]
    int max_pages, num_pages, page_size;
    const int32_t *node_counts;  // per-sequence T_b, or null
    int node_count_add;          // T_b = node_counts[b] + this (1 for a chain's draft lengths)
    StepHook hook;               // fused tree step in cluster mode (step_ctr null otherwise)
    const int32_t *hook_acc;     // the walk's accepted lengths and paths [B, path_stride]
    const int32_t *hook_path;
    int hook_path_stride;
};

sv_status launch_tree_attention(const AttnArgs &args, const AttnPlan &plan, void *ws,
                                cudaStream_t stream);

// ---------------------------------------------------------------- compaction

struct CompactArgs {
    void *k;
    void *v;
    const int32_t *prefix_lens;
    int32_t *new_kv_lens;
    const int32_t *path_nodes;
    int path_stride;
    const int32_t *accepted_len;
    int B, Hkv, D, S_max;  // S_max = max_pages * page_size for a paged cache
    int32_t *seq_status;
    const int32_t *block_table;  // null: contiguous caches [B, Hkv, S_max, D]
    int max_pages, page_size;
    int num_pages;
};

sv_status launch_compact_kv(const CompactArgs &args, cudaStream_t stream);

int device_sm_count();

// Workspace of a fused step: attention, vocabulary pass, then (trees) the
// compaction counters, each 256-byte aligned; 0 if the attention shape is unsupported.
size_t step_workspace_size(bool chain, int B, int T_or_N, int V, int dtype, int Hq, int Hkv,
                           int D);

}  // namespace sv
