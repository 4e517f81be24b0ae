// sv_step.cu -- the fused verification step: one call runs the step's
// attention and its acceptance pass side by side, and folds compaction in.
//
// Source: "Chapitre 9 -- Décodage spéculatif" §9.1: the target's one pass
// over the prefix and the candidates yields the distributions that the
// acceptance then reads, and §9.3: that verification pass is what bounds the
// speed-up.  The attention needs only the K/V caches and Q; the acceptance
// needs only the logits (inputs of the step, already computed), so the two
// share nothing until compaction, which needs both the path and the end of
// the attention's reads.
//
// The caller's stream runs the attention on most of the SMs; a side stream of
// the library's, forked from it and joined back with events, runs the
// vocabulary pass on the rest (the split follows the bytes each side
// streams).  Then:
//   chain: the residual-draw kernel writes the new cache lengths (a chain's
//          accepted rows are already where compaction would put them);
//   tree:  in cluster mode, the last of the attention's row groups and the
//          walk to finish with a (sequence, KV head) moves its path's rows
//          (an arrival counter in the workspace); otherwise a compaction
//          kernel runs after the join.
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "sv_internal.h"

namespace sv {
namespace {

struct SideStream {
    int dev;
    cudaStream_t stream;
    cudaEvent_t fork, join;
};

std::mutex g_side_mu;  // also orders the fork / launch / join sequences of concurrent calls
SideStream g_side[64];
int g_nside = 0;

// The library's side stream and its two events on the current device, made
// by the first step call on that device.  Call with g_side_mu held.
sv_status side_stream(SideStream **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    for (int i = 0; i < g_nside; ++i)
        if (g_side[i].dev == dev) {
            *out = &g_side[i];
            return SV_OK;
        }
    if (g_nside == 64) return SV_ERR_UNSUPPORTED;
    SideStream s{};
    s.dev = dev;
    if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess)
        return SV_ERR_CUDA;
    g_side[g_nside] = s;
    *out = &g_side[g_nside++];
    return SV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CTAs left to the vocabulary side: its share of the step's cost, scaled by
// `boost`, at least 8 and at most half the device.  The costs are bytes (K/V
// taken at the cache capacity S_max, the prefix lengths being device data),
// the attention's multiplied by its row groups (each group streams every
// tile through the tensor cores).  A chain's side ends with the latency-bound
// residual draw, so it needs its statistics done well before the attention:
// boost 1.5 (measured on B=32, N=8, L=4096: the two sides then end
// together); a tree's walk is shorter: 1.3.
int side_ctas(int sms, double attn_cost, double vocab_cost, double boost) {
    int n = (int)std::lround(boost * sms * vocab_cost / (attn_cost + vocab_cost));
    if (n < 8) n = 8;
    if (n > sms / 2) n = sms / 2;
#ifdef SV_PHASE_STAMPS
    // the diagnostic build lets the phase tool try other splits
    if (const char *e = getenv("SV_STEP_SIDE_CTAS")) n = atoi(e);
#endif
    return n;
}

}  // namespace

size_t step_workspace_size(bool chain, int B, int T_or_N, int V, int dtype, int Hq, int Hkv,
                           int D) {
    AttnPlan ap;
    const int T = chain ? T_or_N + 1 : T_or_N;
    if (plan_attention(B, T, Hq, Hkv, D, 1 << 30, &ap) != SV_OK) return 0;
    const VocabPlan vp = plan_vocab(chain, B, T_or_N, V, dtype);
    return align_up(ap.bytes, 256) + align_up(vp.bytes, 256) +
           (chain ? 0 : align_up(sizeof(int) * (size_t)B * Hkv, 256));
}

}  // namespace sv

extern "C" {

sv_status sv_verify_step_chain(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *prefix_lens, int Hq, int Hkv, int D, int S_max,
                               float scale, void *attn_out, int32_t *attn_status,
                               const void *target_logits, const void *draft_logits,
                               sv_dtype dtype, const int32_t *draft_tokens,
                               const int32_t *draft_lens, const float *u_accept,
                               const float *u_sample, int B, int N, int V, int32_t *accepted_len,
                               int32_t *out_tokens, float *probs_out, int32_t *verify_status,
                               int32_t *new_kv_lens, void *workspace, size_t workspace_bytes,
                               sv_stream_t stream) {
    using namespace sv;
    if (!q || !k_cache || !v_cache || !prefix_lens || !attn_out || !target_logits ||
        !draft_logits || !draft_tokens || !u_accept || !u_sample || !accepted_len ||
        !out_tokens || !new_kv_lens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || V <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || S_max < N + 1)
        return SV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !(scale > 0.f) || !std::isfinite(scale)) return SV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(attn_out) ||
        !aligned16(target_logits) || !aligned16(draft_logits))
        return SV_ERR_INVALID_ARG;
    // the attention reads the prefix lengths while the acceptance writes the new ones
    if (new_kv_lens == prefix_lens) return SV_ERR_INVALID_ARG;
    if ((long long)B * Hkv * S_max >= (1LL << 31) || N > 63 || V >= (1 << 30))
        return SV_ERR_UNSUPPORTED;
    const int T = N + 1;
    const int sms = device_sm_count();
    if (sms <= 0) return SV_ERR_CUDA;
    const int esz = dtype == SV_F32 ? 4 : 2;
    const int side = side_ctas(sms, 4.0 * B * Hkv * (double)S_max * D,
                               (double)B * (2 * N + 1) * V * esz, 1.5);
    AttnPlan ap;
    sv_status st = plan_attention(B, T, Hq, Hkv, D, S_max, &ap, sms - side);
    if (st != SV_OK) return st;
    VocabPlan vp = plan_vocab(true, B, N, V, dtype);
    if ((size_t)B * vp.rows_per_seq * vp.nchunks >= (1u << 31) || vp.res_chunks > kMaxResChunks)
        return SV_ERR_UNSUPPORTED;
    vp.max_ctas = sms - ap.grid;
    const size_t off_v = align_up(ap.bytes, 256);
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < off_v + align_up(vp.bytes, 256))
        return SV_ERR_WORKSPACE;

    AttnArgs aa{};
    aa.q = q;
    aa.k = k_cache;
    aa.v = v_cache;
    aa.prefix_lens = prefix_lens;
    aa.parents = nullptr;  // a chain: the causal mask
    aa.B = B;
    aa.T = T;
    aa.Hq = Hq;
    aa.Hkv = Hkv;
    aa.D = D;
    aa.S_max = S_max;
    aa.scale = scale;
    aa.out = attn_out;
    aa.seq_status = attn_status;
    aa.node_counts = draft_lens;  // N_b drafts: N_b + 1 nodes
    aa.node_count_add = 1;
    ChainArgs ca{};
    ca.target = target_logits;
    ca.draft = draft_logits;
    ca.tokens = draft_tokens;
    ca.draft_lens = draft_lens;
    ca.u_accept = u_accept;
    ca.u_sample = u_sample;
    ca.B = B;
    ca.N = N;
    ca.V = V;
    ca.accepted_len = accepted_len;
    ca.out_tokens = out_tokens;
    ca.probs = probs_out;
    ca.seq_status = verify_status;
    ca.prefix_lens = prefix_lens;
    ca.new_kv_lens = new_kv_lens;
    ca.S_max = S_max;

    cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream *sd = nullptr;
    if ((st = side_stream(&sd)) != SV_OK) return st;
    if (cudaEventRecord(sd->fork, main) != cudaSuccess ||
        cudaStreamWaitEvent(sd->stream, sd->fork, 0) != cudaSuccess)
        return SV_ERR_CUDA;
    // the attention first, so that its CTAs (clusters, in cluster mode) are
    // placed before the vocabulary pass takes the SMs left to it
    const sv_status st2 = launch_tree_attention(aa, ap, workspace, main);
    st = launch_verify_chain(ca, dtype, vp, static_cast<char *>(workspace) + off_v, sd->stream);
    // join even after a failed launch, so the caller's stream never runs ahead
    if (cudaEventRecord(sd->join, sd->stream) != cudaSuccess ||
        cudaStreamWaitEvent(main, sd->join, 0) != cudaSuccess)
        return SV_ERR_CUDA;
    return st != SV_OK ? st : st2;
}

sv_status sv_verify_step_tree_greedy(const void *q, void *k_cache, void *v_cache,
                                     const int32_t *prefix_lens, const int32_t *parents,
                                     const int32_t *node_counts, int B, int T, int Hq, int Hkv,
                                     int D, int S_max, float scale, void *attn_out,
                                     int32_t *attn_status, const void *target_logits,
                                     sv_dtype dtype, const int32_t *node_tokens, int V,
                                     int32_t *accepted_len, int32_t *path_nodes,
                                     int32_t *out_tokens, int32_t *verify_status,
                                     int32_t *new_kv_lens, void *workspace,
                                     size_t workspace_bytes, sv_stream_t stream) {
    using namespace sv;
    if (!q || !k_cache || !v_cache || !prefix_lens || !attn_out || !target_logits ||
        !node_tokens || !accepted_len || !path_nodes || !out_tokens || !new_kv_lens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || V <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || S_max < T)
        return SV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !(scale > 0.f) || !std::isfinite(scale)) return SV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(attn_out) ||
        !aligned16(target_logits))
        return SV_ERR_INVALID_ARG;
    if (new_kv_lens == prefix_lens) return SV_ERR_INVALID_ARG;
    if ((long long)B * Hkv * S_max >= (1LL << 31) || V >= (1 << 30) || Hkv > 256)
        return SV_ERR_UNSUPPORTED;
    const int sms = device_sm_count();
    if (sms <= 0) return SV_ERR_CUDA;
    const int esz = dtype == SV_F32 ? 4 : 2;
    // Attention first: in cluster mode it takes the CTAs its clusters need
    // (leaving at least 8 SMs), in the flat split its share of the cost.
    // With several row groups per KV head in the flat split (the EAGLE-size
    // trees: 256 query rows per KV head) the attention is paced by its tensor
    // and softmax work, not by HBM, so SMs taken from it cost more than the
    // overlap gives back (B=16, T=64, L=8192: 192 us side by side, 187 us one
    // kernel after another): there the kernels run in sequence on the
    // caller's stream, each with the whole device.
    AttnPlan ap;
    sv_status st = plan_attention(B, T, Hq, Hkv, D, S_max, &ap, sms - 8);
    if (st != SV_OK) return st;
    const bool serial = ap.cluster <= 1 && ap.rg >= 2;
    if (serial) {
        if ((st = plan_attention(B, T, Hq, Hkv, D, S_max, &ap)) != SV_OK) return st;
    } else if (ap.cluster <= 1) {
        const int side = side_ctas(sms, 4.0 * B * Hkv * (double)S_max * D * ap.rg,
                                   (double)B * T * V * esz, 1.3);
        if ((st = plan_attention(B, T, Hq, Hkv, D, S_max, &ap, sms - side)) != SV_OK) return st;
    }
    VocabPlan vp = plan_vocab(false, B, T, V, dtype);
    if ((size_t)B * vp.rows_per_seq * vp.nchunks >= (1u << 31)) return SV_ERR_UNSUPPORTED;
    vp.max_ctas = serial ? 0 : sms - ap.grid;
    const size_t off_v = align_up(ap.bytes, 256);
    const size_t off_c = off_v + align_up(vp.bytes, 256);
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < off_c + align_up(sizeof(int) * (size_t)B * Hkv, 256))
        return SV_ERR_WORKSPACE;
    // compaction inside the two kernels when the attention runs in clusters and
    // the walk in a kernel of its own (rows 16-byte aligned), for at most
    // kStepHookMaxT nodes; else a kernel after both (in the serial order too:
    // the walk moving the rows alone, one sequence a CTA, measured 3 us slower
    // than the compaction kernel on the EAGLE step)
    const bool hook = ap.cluster > 1 && vp.vec && D == 128 && T <= kStepHookMaxT;

    StepHook hk{};
    if (hook) {
        hk.step_ctr = reinterpret_cast<int *>(static_cast<char *>(workspace) + off_c);
        hk.k = static_cast<uint4 *>(k_cache);
        hk.v = static_cast<uint4 *>(v_cache);
        hk.prefix_lens = prefix_lens;
        hk.new_kv_lens = new_kv_lens;
        hk.Hkv = Hkv;
        hk.rg_count = ap.rg;
        hk.S_max = S_max;
        hk.D = D;
    }
    AttnArgs aa{};
    aa.q = q;
    aa.k = k_cache;
    aa.v = v_cache;
    aa.prefix_lens = prefix_lens;
    aa.parents = parents;
    aa.B = B;
    aa.T = T;
    aa.Hq = Hq;
    aa.Hkv = Hkv;
    aa.D = D;
    aa.S_max = S_max;
    aa.scale = scale;
    aa.out = attn_out;
    aa.seq_status = attn_status;
    aa.node_counts = node_counts;
    aa.hook = hk;
    aa.hook_acc = accepted_len;
    aa.hook_path = path_nodes;
    aa.hook_path_stride = T;
    TreeArgs ta{};
    ta.target = target_logits;
    ta.tokens = node_tokens;
    ta.parents = parents;
    ta.node_counts = node_counts;
    ta.B = B;
    ta.T = T;
    ta.V = V;
    ta.accepted_len = accepted_len;
    ta.path_nodes = path_nodes;
    ta.out_tokens = out_tokens;
    ta.seq_status = verify_status;
    ta.hook = hk;

    cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
    if (serial) {
        // one kernel after another (programmatic launch chains them)
        if ((st = launch_tree_attention(aa, ap, workspace, main)) != SV_OK) return st;
        if ((st = launch_verify_tree_greedy(ta, dtype, vp, static_cast<char *>(workspace) + off_v,
                                            main)) != SV_OK)
            return st;
    } else {
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *sd = nullptr;
        if ((st = side_stream(&sd)) != SV_OK) return st;
        if (cudaEventRecord(sd->fork, main) != cudaSuccess ||
            cudaStreamWaitEvent(sd->stream, sd->fork, 0) != cudaSuccess)
            return SV_ERR_CUDA;
        const sv_status st2 = launch_tree_attention(aa, ap, workspace, main);
        st = launch_verify_tree_greedy(ta, dtype, vp, static_cast<char *>(workspace) + off_v,
                                       sd->stream);
        if (cudaEventRecord(sd->join, sd->stream) != cudaSuccess ||
            cudaStreamWaitEvent(main, sd->join, 0) != cudaSuccess)
            return SV_ERR_CUDA;
        if (st != SV_OK) return st;
        if (st2 != SV_OK) return st2;
    }
    if (hook) return SV_OK;
    CompactArgs c{};
    c.k = k_cache;
    c.v = v_cache;
    c.prefix_lens = prefix_lens;
    c.new_kv_lens = new_kv_lens;
    c.path_nodes = path_nodes;
    c.path_stride = T;
    c.accepted_len = accepted_len;
    c.B = B;
    c.Hkv = Hkv;
    c.D = D;
    c.S_max = S_max;
    c.seq_status = nullptr;  // a bad path is already reported by the acceptance
    return launch_compact_kv(c, main);
}

}  // extern "C"
