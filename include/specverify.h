/*
 * specverify.h -- C ABI of libspecverify: the target model's verification
 * step of speculative decoding, on one GPU (sm_103a).
 *
 * The step, as the source pages state it ("Chapitre 9 -- Décodage
 * spéculatif", LLM Primer VI, §9.1-§9.2; "Parallel Decoding" glossary,
 * Medusa "Tree attention", "L'attention en arbre : la brique commune" and
 * "Limites du parallel decoding"):
 *   1. one attention pass in which N+1 chain positions, or T draft-tree
 *      nodes, attend to the prefix KV cache plus their own tree ancestors
 *      (sv_tree_attention);
 *   2. acceptance over the full vocabulary: stochastic min(1, p(x)/q(x))
 *      with a residual (p-q)+ resample and a bonus token on chains
 *      (sv_verify_chain), greedy longest agreeing path on trees
 *      (sv_verify_tree_greedy);
 *   3. compaction of the accepted path's K/V rows (sv_compact_kv).
 *
 * Conventions shared by every call:
 *   - Every array argument is DEVICE memory owned by the caller.  The
 *     library allocates nothing and, apart from the fixed scratch array of
 *     sv_verify_chain_noalloc, keeps no state between calls.  Calls
 *     that need scratch take a caller-provided workspace; its size comes
 *     from sv_workspace_size() and it must be zero-filled once before its
 *     first use (every call leaves its counters at zero again; after a call
 *     that reported SV_ERR_TIMEOUT, zero-fill it again).
 *   - Every call is asynchronous on `stream` (NULL = legacy default
 *     stream); none synchronises.  Two calls that share a workspace must
 *     not overlap on the GPU.
 *   - Host-detectable errors (bad sizes, NULL pointers, misalignment,
 *     workspace too small, unsupported shape) return a non-OK status before
 *     anything is launched.  Problems only visible on the device (a parent
 *     array that is not a topologically ordered tree, a token outside
 *     [0, V), prefix_len + T > S_max, a logits row whose max or normaliser is
 *     not finite) are reported per sequence in seq_status[b] (nullable);
 *     such a sequence's outputs are -1 (token/length outputs) or left
 *     unspecified (attention rows).  No call ever traps the GPU.
 *   - Layouts are dense row-major with the innermost dimension last.  bf16
 *     is IEEE binary32's upper 16 bits.  Pointers to bf16/f32 tensors must
 *     be 16-byte aligned.
 *   - Tree convention: node 0 is the root (the last committed token, whose
 *     K/V this pass produces); parents[b][0] = -1 and 0 <= parents[b][i] < i.
 *     A chain of N drafts is the tree parent[i] = i-1 with T = N+1 nodes.
 *     Node j's K/V row sits in cache slot prefix_lens[b] + j.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared opaquely so that this header needs no CUDA headers. */
typedef struct CUstream_st *sv_stream_t;

typedef enum sv_status {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,  /* host: NULL pointer, size <= 0, misaligned pointer, Hq % Hkv */
    SV_ERR_WORKSPACE = 2,    /* host: workspace NULL or smaller than sv_workspace_size()  */
    SV_ERR_UNSUPPORTED = 3,  /* host: shape outside the kernels' range (see each call)    */
    SV_ERR_CUDA = 4,         /* host: a CUDA runtime call or launch failed                 */
    SV_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel gave up             */
    SV_ERR_BAD_INPUT = 6     /* device: invalid per-sequence data (see conventions)       */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum sv_op {
    SV_OP_TREE_ATTENTION = 0,
    SV_OP_VERIFY_CHAIN = 1,
    SV_OP_VERIFY_TREE_GREEDY = 2,
    SV_OP_VERIFY_TREE_STOCHASTIC = 3,
    SV_OP_VERIFY_STEP_CHAIN = 4,
    SV_OP_VERIFY_STEP_TREE_GREEDY = 5
} sv_op;

/*
 * Bytes of workspace a call needs, for the CURRENT device (the kernels size
 * their persistent grids by its SM count).  Arguments are those of the call;
 * the ones an operation does not use are ignored:
 *   SV_OP_TREE_ATTENTION:          B, T, Hq, Hkv, D
 *   SV_OP_VERIFY_CHAIN:            B, N (as T_or_N), V, dtype
 *   SV_OP_VERIFY_TREE_GREEDY:      B, T, V, dtype
 *   SV_OP_VERIFY_TREE_STOCHASTIC:  B, T, V, dtype
 *   SV_OP_VERIFY_STEP_CHAIN:       B, N (as T_or_N), V, dtype, Hq, Hkv, D
 *   SV_OP_VERIFY_STEP_TREE_GREEDY: B, T, V, dtype, Hq, Hkv, D
 * Returns 0 for invalid arguments and for shapes the call refuses as
 * SV_ERR_UNSUPPORTED.
 */
size_t sv_workspace_size(sv_op op, int B, int T_or_N, int V, sv_dtype dtype, int Hq, int Hkv,
                         int D);

/*
 * Verification attention over a prefix KV cache plus each node's ancestors.
 * Source: "Chapitre 9 -- Décodage spéculatif" §9.1 (one forward over the
 * prefix concatenated with the N candidates yields N+1 distributions, and
 * stays memory-bound) and §9.2 (EAGLE-2's draft tree verified in one
 * attention pass with a custom mask); "Parallel Decoding" glossary, Medusa
 * "Tree attention" and "L'attention en arbre" (all branches scored in one
 * pass under a mask encoding the tree).
 *
 * For sequence b, node t, query head h (KV head h / (Hq/Hkv)):
 *   out[b,t,h,:] = sum_j softmax_j(scale * q[b,t,h,:] . k_j) v_j
 * over cache slots j in [0, L_b) and L_b + i for every node i on the
 * root->t path (t included), L_b = prefix_lens[b].
 *
 *   q           bf16 [B, T, Hq, D]
 *   k_cache     bf16 [B, Hkv, S_max, D]; v_cache likewise.  Slots at and
 *               beyond L_b + T are never read (they may hold anything).
 *   prefix_lens int32 [B]; each 0 <= L_b and L_b + T <= S_max (else
 *               seq_status[b] = SV_ERR_BAD_INPUT and the sequence is skipped)
 *   parents     int32 [B, T] parent array, or NULL for a chain (causal mask)
 *   node_counts int32 [B] or NULL: sequence b has T_b nodes (1 <= T_b <= T;
 *               a variable-length batch), nodes t >= T_b are padding -- their
 *               output rows are left unspecified and their slots unread, and
 *               L_b + T_b replaces L_b + T above; NULL means T_b = T
 *   scale       > 0 and finite, normally 1/sqrt(D)
 *   out         bf16 [B, T, Hq, D]
 *   seq_status  int32 [B] or NULL
 *   workspace   >= sv_workspace_size(SV_OP_TREE_ATTENTION, ...) bytes
 * Supported: D = 128, 1 <= T <= 64, Hq % Hkv == 0, Hq/Hkv * T <= 512,
 * B <= 4096, B * Hkv * S_max < 2^31.
 */
sv_status sv_tree_attention(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *prefix_lens, const int32_t *parents,
                            const int32_t *node_counts, int B, int T, int Hq, int Hkv, int D,
                            int S_max, float scale, void *out, int32_t *seq_status,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream);

/*
 * Verification attention over a paged KV cache (the paged KV of "Chapitre 9",
 * section "Ce que prépare le Chapitre 9": the cache held in fixed-size pages
 * reached through a per-sequence page table).  The same computation as sv_tree_attention, with logical slot s of
 * sequence b (prefix slots 0..L_b-1, node j at slot L_b + j) stored in page
 * block_table[b][s / page_size] at offset s % page_size.
 *
 *   k_pages, v_pages  bf16 [num_pages, Hkv, page_size, D]
 *   block_table       int32 [B, max_pages]: physical page of each logical page
 *   other arguments   as sv_tree_attention, with S_max = max_pages * page_size
 *   workspace         >= sv_workspace_size(SV_OP_TREE_ATTENTION, ...) bytes
 * Supported: page_size a power of two >= 8 or a multiple of 128;
 * num_pages * Hkv * page_size < 2^31; otherwise as sv_tree_attention.  A
 * page id outside [0, num_pages) among the pages that hold slots
 * [0, L_b + T) is reported as SV_ERR_BAD_INPUT for that sequence (its
 * rows read as zeros); entries past those pages are never used.
 */
sv_status sv_tree_attention_paged(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *block_table, int max_pages, int num_pages,
                                  int page_size, const int32_t *prefix_lens,
                                  const int32_t *parents, const int32_t *node_counts, int B,
                                  int T, int Hq, int Hkv, int D, float scale, void *out,
                                  int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                  sv_stream_t stream);

/*
 * Stochastic chain acceptance over the full vocabulary.
 * Source: "Chapitre 9 -- Décodage spéculatif" §9.1: the target yields a
 * distribution at each of the N+1 positions; draft token x drawn from q is
 * accepted with probability min(1, p(x)/q(x)), else a token is drawn from the
 * normalised residual (p-q)+; the output is then distributed exactly as the
 * target's own sampling.  The bonus token after N acceptances is drawn from
 * the (N+1)-th distribution.
 *
 * Per sequence b, with p_i = softmax(target[b,i,:]), q_i = softmax(draft[b,i,:]):
 *   accept_i  <=>  u_accept[b,i] * q_i(x_i) < p_i(x_i)
 *   a = first i with !accept_i, or N
 *   r = max(0, p_a - q_a) if a < N (p_a itself if that sums to 0), r = p_N if a = N
 *   y = min{k : r_0 + ... + r_k > u_sample[b] * sum(r)}   (index order)
 *   accepted_len[b] = a; out_tokens[b,:] = x_0..x_{a-1}, y, then -1 padding
 *
 *   target_logits  [B, N+1, V] of `dtype`, already temperature-scaled
 *   draft_logits   [B, N, V] of `dtype`
 *   draft_tokens   int32 [B, N]
 *   draft_lens     int32 [B] or NULL: sequence b drafted N_b tokens
 *                  (0 <= N_b <= N; a variable-length batch): positions and
 *                  rows past N_b are padding, the bonus after N_b acceptances
 *                  comes from target row N_b, out_tokens holds N_b + 1 entries
 *                  then -1, probs_out is 0 past N_b; NULL means N_b = N
 *   u_accept       f32 [B, N] uniforms in [0, 1); u_sample f32 [B]
 *   accepted_len   int32 [B];  out_tokens int32 [B, N+1]
 *   probs_out      f32 [B, N, 2] = (p_i(x_i), q_i(x_i)) for every i, or NULL
 * Supported: 1 <= N <= 63, 1 <= V < 2^30, dtype SV_F32 or SV_BF16.
 * Launches two kernels (row statistics, then the decisions and the residual
 * draw).  If a bounded wait of the statistics pass gives up, every sequence
 * of the call reports SV_ERR_TIMEOUT (outputs -1).
 */
sv_status sv_verify_chain(const void *target_logits, const void *draft_logits, sv_dtype dtype,
                          const int32_t *draft_tokens, const int32_t *draft_lens,
                          const float *u_accept, const float *u_sample, int B, int N, int V,
                          int32_t *accepted_len, int32_t *out_tokens, float *probs_out,
                          int32_t *seq_status, void *workspace, size_t workspace_bytes,
                          sv_stream_t stream);

/*
 * Greedy longest-agreeing-path acceptance on a draft tree.
 * Source: "Parallel Decoding" glossary, "L'attention en arbre": the longest
 * accepted path becomes the generated sequence; "Chapitre 9" §9.1: the
 * longest prefix on which the candidates agree with the target is kept and
 * at the divergence the engine takes the target's own choice.
 *
 *   am_i = argmax_v target[b,i,v] (smallest v among equal maxima)
 *   ok_0 = 1; ok_i = ok_{parent_i} and node_tokens[b,i] == am_{parent_i}
 *   d* = deepest ok node (smallest index among equal depths)
 *   accepted_len[b] = depth(d*); path_nodes[b,:] = root..d* then -1;
 *   out_tokens[b,:] = node_tokens of path nodes 1..depth, am_{d*}, then -1
 *
 *   target_logits [B, T, V] of `dtype`; node_tokens, parents int32 [B, T]
 *   node_counts int32 [B] or NULL: sequence b has T_b nodes (1 <= T_b <= T),
 *   those past T_b are padding and never accepted; NULL means T_b = T
 *   (parents NULL: a chain, parent_i = i - 1, i.e. greedy chain
 *   verification -- the longest prefix of draft tokens each equal to the
 *   target's argmax at the position before it, then that argmax)
 *   accepted_len int32 [B]; path_nodes, out_tokens int32 [B, T]
 * Supported: 1 <= T <= 1024, 1 <= V < 2^30.
 */
sv_status sv_verify_tree_greedy(const void *target_logits, sv_dtype dtype,
                                const int32_t *node_tokens, const int32_t *parents,
                                const int32_t *node_counts, int B, int T, int V,
                                int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                                int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                sv_stream_t stream);

/*
 * Stochastic acceptance on a draft tree: multi-draft speculative sampling.
 * Source: "Chapitre 9 -- Décodage spéculatif" §9.2 has the target choose
 * among several drafted paths (EAGLE-2's tree) but gives no rule; the rule
 * here is the one of SpecInfer (Miao et al., ASPLOS 2024).  Node u's children
 * were drawn independently from the draft's distribution at u,
 * q_u = softmax(draft[b,u,:]); the target's is p_u = softmax(target[b,u,:]).
 *
 * From the root, at node u with c = 0:
 *   N(c) = sum_v max(0, p_u(v) - c q_u(v))          (1 for c = 0)
 *   for the children v of u in index order, x = node_tokens[b,v]:
 *     accept v  <=>  u_accept[b,v] * q_u(x) * N(c) < max(0, p_u(x) - c q_u(x))
 *     accepted: the walk moves to v (c = 0 there); rejected: c = c + N(c)
 *   no child accepted, or u a leaf: y drawn from the weights max(0, p_u - c q_u)
 *   (p_u if they sum to 0) by y = min{k : w_0 + ... + w_k > u_sample[b] * sum(w)}
 * (the rejection step of speculative sampling applied to the current residual
 * r_c = max(0, p_u - c q_u) / N(c), in closed form).  A chain-shaped tree is
 * the chain rule of sv_verify_chain.
 *   accepted_len[b] = depth of the last accepted node; path_nodes[b,:] = root..it,
 *   then -1; out_tokens[b,:] = tokens of path nodes 1..depth, y, then -1
 *
 *   target_logits, draft_logits [B, T, V] of `dtype`, temperature-scaled
 *                  (draft row u: the distribution u's children came from;
 *                  rows of leaves are not read)
 *   node_tokens, parents int32 [B, T] (parents NULL: a chain); u_accept f32
 *   [B, T] (entry v tests node v; entry 0 unused); u_sample f32 [B]
 *   node_counts int32 [B] or NULL: sequence b has T_b nodes (1 <= T_b <= T),
 *   those past T_b are padding (never read); NULL means T_b = T
 *   accepted_len int32 [B]; path_nodes, out_tokens int32 [B, T]
 *   workspace  >= sv_workspace_size(SV_OP_VERIFY_TREE_STOCHASTIC, B, T, V, dtype, 0, 0)
 * Supported: 1 <= T <= 1024, 1 <= V <= 2^22.  A tree that is not
 * topologically ordered, a token outside [0, V) or a used row without a
 * finite distribution is reported as SV_ERR_BAD_INPUT for its sequence.
 * Each rejected sibling costs one pass over its node's row pair.
 */
sv_status sv_verify_tree_stochastic(const void *target_logits, const void *draft_logits,
                                    sv_dtype dtype, const int32_t *node_tokens,
                                    const int32_t *parents, const int32_t *node_counts,
                                    const float *u_accept, const float *u_sample, int B, int T,
                                    int V,
                                    int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                                    int32_t *seq_status, void *workspace, size_t workspace_bytes,
                                    sv_stream_t stream);

/*
 * Compaction of the accepted path's rows in the enlarged KV cache.
 * Source: "Parallel Decoding" glossary, "Limites du parallel decoding" (tree
 * attention needs a KV cache enlarged for the branches); "Chapitre 9" §9.1
 * (the accepted prefix is kept and the rest discarded).
 *
 * In place, per sequence b with a = accepted_len[b] >= 0, L = prefix_lens[b]:
 *   for d = 0..a, every KV head: row L + d <- row L + path[d]
 *   new_kv_lens[b] = L + a + 1
 * path[d] = path_nodes[b * path_stride + d], or d when path_nodes is NULL
 * (a chain: nothing moves).  A path must start at 0 and increase strictly
 * (so path[d] >= d) with L + path[a] < S_max, a < path_stride and
 * L + a + 1 <= S_max; otherwise nothing moves, new_kv_lens[b] = L and
 * seq_status[b] = SV_ERR_BAD_INPUT.  A negative accepted_len (an upstream
 * error) leaves the sequence untouched with new_kv_lens[b] = L.
 * new_kv_lens may alias prefix_lens.
 *
 *   k_cache, v_cache bf16 [B, Hkv, S_max, D]
 * Supported: D % 8 == 0, D <= 256.
 */
sv_status sv_compact_kv(void *k_cache, void *v_cache, const int32_t *prefix_lens,
                        int32_t *new_kv_lens, const int32_t *path_nodes, int path_stride,
                        const int32_t *accepted_len, int B, int Hkv, int D, int S_max,
                        int32_t *seq_status, sv_stream_t stream);

/*
 * Compaction of the accepted path's rows in a paged KV cache: sv_compact_kv
 * with rows addressed through the page table (layout as in
 * sv_tree_attention_paged, S_max = max_pages * page_size).  A page id
 * outside [0, num_pages) for a slot the move reads or writes makes the
 * sequence SV_ERR_BAD_INPUT with nothing moved.
 */
sv_status sv_compact_kv_paged(void *k_pages, void *v_pages, const int32_t *block_table,
                              int max_pages, int num_pages, int page_size,
                              const int32_t *prefix_lens, int32_t *new_kv_lens,
                              const int32_t *path_nodes, int path_stride,
                              const int32_t *accepted_len, int B, int Hkv, int D,
                              int32_t *seq_status, sv_stream_t stream);

/*
 * The fused verification step on a chain: sv_tree_attention with the causal
 * mask, sv_verify_chain and the compaction of the accepted rows, in one call.
 * Source: "Chapitre 9 -- Décodage spéculatif" §9.1 (one pass over the prefix
 * and the N candidates yields the N+1 distributions the acceptance reads;
 * the accepted prefix is kept) and §9.3 (the verification pass bounds the
 * speed-up).  The logits are inputs, so the attention and the acceptance are
 * independent: the attention runs on the caller's stream over most of the
 * SMs while the acceptance runs on the rest, on a side stream of the library
 * forked from `stream` and joined back to it (two events); the SMs are split
 * in proportion to the bytes each side streams.  A chain's accepted rows are
 * already in place (node d at slot L_b + d), so compaction writes only the
 * new cache lengths.
 *
 * Arguments as sv_tree_attention (parents = NULL; node counts N_b + 1 from
 * draft_lens) and sv_verify_chain, plus
 *   attn_status    int32 [B] or NULL: sv_tree_attention's seq_status
 *   verify_status  int32 [B] or NULL: sv_verify_chain's seq_status
 *   new_kv_lens    int32 [B]: L_b + a_b + 1, or L_b when a_b < 0 or
 *                  L_b + N_b + 1 > S_max; must not alias prefix_lens (the
 *                  attention reads those while the acceptance writes these)
 *   workspace      >= sv_workspace_size(SV_OP_VERIFY_STEP_CHAIN, B, N, V,
 *                  dtype, Hq, Hkv, D) bytes, zero-filled before its first use
 * Supported: as the two calls.  The first step call on a device creates the
 * side stream and events (make it before any stream capture); calls from
 * several host threads are serialised around the fork and the join.
 */
sv_status sv_verify_step_chain(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *prefix_lens, int Hq, int Hkv, int D, int S_max,
                               float scale, void *attn_out, int32_t *attn_status,
                               const void *target_logits, const void *draft_logits,
                               sv_dtype dtype, const int32_t *draft_tokens,
                               const int32_t *draft_lens, const float *u_accept,
                               const float *u_sample, int B, int N, int V, int32_t *accepted_len,
                               int32_t *out_tokens, float *probs_out, int32_t *verify_status,
                               int32_t *new_kv_lens, void *workspace, size_t workspace_bytes,
                               sv_stream_t stream);

/*
 * The fused verification step on a draft tree: sv_tree_attention,
 * sv_verify_tree_greedy and sv_compact_kv in one call.  Sources as those
 * three calls and sv_verify_step_chain.  The attention and the greedy
 * acceptance run side by side as in sv_verify_step_chain, except when the
 * attention has several row groups per KV head (Hq/Hkv * T > 128) and too many
 * of them for cluster mode: then it is paced by its own tensor and softmax
 * work, and the kernels run one after another, each with the whole device.
 * When the attention runs in cluster mode (few row groups: B * Hkv *
 * ceil(Hq/Hkv * T / 128) clusters fit on the device at once) and the logits
 * rows are 16-byte aligned, compaction happens inside the two kernels: for
 * each (sequence, KV head), whichever of the attention (done reading that
 * head's rows) and the tree walk (path known) arrives last moves the rows.
 * Otherwise a compaction kernel runs after both.
 *
 * Arguments as the three calls (path_nodes has T columns), plus attn_status,
 * verify_status (nullable, as above) and
 *   k_cache, v_cache  read by the attention, then compacted in place
 *   new_kv_lens       int32 [B]: L_b + a_b + 1, or L_b when a_b < 0 or the
 *                     cache cannot hold the nodes; must not alias prefix_lens
 *   workspace         >= sv_workspace_size(SV_OP_VERIFY_STEP_TREE_GREEDY, B,
 *                     T, V, dtype, Hq, Hkv, D) bytes, zero-filled before first use
 * Supported: as the three calls, with Hkv <= 256.
 */
sv_status sv_verify_step_tree_greedy(const void *q, void *k_cache, void *v_cache,
                                     const int32_t *prefix_lens, const int32_t *parents,
                                     const int32_t *node_counts, int B, int T, int Hq, int Hkv,
                                     int D, int S_max, float scale, void *attn_out,
                                     int32_t *attn_status, const void *target_logits,
                                     sv_dtype dtype, const int32_t *node_tokens, int V,
                                     int32_t *accepted_len, int32_t *path_nodes,
                                     int32_t *out_tokens, int32_t *verify_status,
                                     int32_t *new_kv_lens, void *workspace,
                                     size_t workspace_bytes, sv_stream_t stream);

/*
 * Chain acceptance with no caller workspace.  There is no counterpart of this
 * call in the source pages: it is a deployment convenience.
 *
 * Some callers cannot hand the library a workspace because they cannot
 * allocate device memory where they call it: a plugin whose host has given
 * all device memory to its own pool and exposes no allocator, or a real-time
 * loop that must not take the device-wide synchronisation cudaMalloc and
 * cudaFree imply.  This call computes what sv_verify_chain computes with
 * draft_lens = NULL (every sequence drafted all N tokens; a ragged batch
 * goes through sv_verify_chain), with the same kernels and outputs, but keeps
 * its scratch in a fixed array inside the library, SV_NOALLOC_SCRATCH_BYTES
 * long.  Every GPU that loads the library holds that array until the process
 * exits.
 *
 * - It calls no cudaMalloc, cudaFree or other allocating routine.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it for the
 *   life of the process: call it in the device's primary context, and not
 *   after a cudaDeviceReset of that device.
 * - All calls share the one array, which keeps the last call's contents; each
 *   call clears the part that must start at zero (cudaMemsetAsync on
 *   `stream`).  Calls that overlap on the GPU (other streams, other host
 *   threads) race on the array and give wrong results: serialise them.
 * - Returns SV_ERR_WORKSPACE, launching nothing, when the scratch this shape
 *   needs (sv_workspace_size(SV_OP_VERIFY_CHAIN, ...)) exceeds
 *   SV_NOALLOC_SCRATCH_BYTES; the other errors are those of sv_verify_chain.
 */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)

sv_status sv_verify_chain_noalloc(const void *target_logits, const void *draft_logits,
                                  sv_dtype dtype, const int32_t *draft_tokens,
                                  const float *u_accept, const float *u_sample, int B, int N,
                                  int V, int32_t *accepted_len, int32_t *out_tokens,
                                  float *probs_out, int32_t *seq_status, sv_stream_t stream);

/* Static, human-readable name of a status code. */
const char *sv_status_string(sv_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
