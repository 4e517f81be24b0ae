/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the target model's
 * verification step of speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library; both sides only see the same seeded input bytes.
 *
 * Every function evaluates the definition it cites directly, in double
 * precision, in index order, with no blocking, fusion or reordering:
 *
 *   - tree / chain verification attention  ("Parallel Decoding" glossary,
 *     "L'attention en arbre : la brique commune"; Medusa "Tree attention";
 *     "Chapitre 9 -- Décodage spéculatif" §9.1 and §9.2),
 *   - full-vocabulary softmax statistics and the stochastic acceptance rule
 *     min(1, p(x)/q(x)) with the normalised residual (p-q)+ and the bonus
 *     token drawn from the (N+1)-th distribution (Chapitre 9 §9.1),
 *   - greedy longest-agreeing-path acceptance on a draft tree (glossary,
 *     "L'attention en arbre"; Chapitre 9 §9.1, the longest agreeing prefix),
 *   - stochastic acceptance on a draft tree (Chapitre 9 §9.2 has the target
 *     choose among several drafted paths but gives no rule; the rule here is
 *     the multi-draft speculative sampling of SpecInfer, Miao et al. 2024),
 *   - compaction of the accepted path's K/V rows ("Parallel Decoding",
 *     "Limites du parallel decoding": the enlarged KV cache for branches).
 *
 * Readings of points the pages leave open are listed in the design notes and
 * restated at each function.  Status codes are this file's own numbers; they
 * happen to match the library's public enum so tests can compare them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    ORC_OK = 0,
    ORC_ERR_INVALID_ARG = 1,
    ORC_ERR_BAD_INPUT = 6
};

/* flag bits written per sequence by the acceptance oracles */
enum {
    ORC_FLAG_ACCEPT_NEAR_TIE = 1,   /* |u*q(x) - p(x)| < 1e-6 * p(x) at a decision taken */
    ORC_FLAG_SAMPLE_NEAR_TIE = 2,   /* u*S within 1e-6*S of a cumulative-sum boundary   */
    ORC_FLAG_DEGENERATE_RESIDUAL = 4 /* (p-q)+ summed to zero: sampled from p instead    */
};

/* ---- element access -------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* dtype 0 = float32, 1 = bf16 (stored as raw uint16 bits) */
static double logit_at(const void *base, int dtype, size_t idx)
{
    if (dtype == 0)
        return (double)((const float *)base)[idx];
    return bf16_bits_to_double(((const uint16_t *)base)[idx]);
}

/* ---- A1: ancestor mask ------------------------------------------------- */

/*
 * Tree structure as a parent array (glossary "L'attention en arbre": the root
 * is the last verified token and the mask encodes the tree).  Reading: node 0
 * is the root with parents[0] == -1 and every other node's parent precedes it
 * (0 <= parents[i] < i).  parents == NULL means a chain, parent[i] = i-1.
 *
 * mask[t*T + j] = 1 iff node j lies on the root->t path (t itself included),
 * found by walking parent pointers from t up to the root.  depth[t] counts the
 * edges on that path.  Returns ORC_ERR_BAD_INPUT for an invalid parent array.
 */
int orc_ancestor_mask(const int32_t *parents, int T, uint8_t *mask, int32_t *depth)
{
    if (T <= 0)
        return ORC_ERR_INVALID_ARG;
    if (parents) {
        if (parents[0] != -1)
            return ORC_ERR_BAD_INPUT;
        for (int i = 1; i < T; ++i)
            if (parents[i] < 0 || parents[i] >= i)
                return ORC_ERR_BAD_INPUT;
    }
    memset(mask, 0, (size_t)T * (size_t)T);
    for (int t = 0; t < T; ++t) {
        int node = t, edges = 0;
        for (;;) {
            mask[(size_t)t * T + node] = 1;
            int up = parents ? parents[node] : node - 1;
            if (up < 0)
                break;
            node = up;
            ++edges;
        }
        if (depth)
            depth[t] = edges;
    }
    return ORC_OK;
}

/* ---- A2: verification attention ---------------------------------------- */

/*
 * One forward over the prefix concatenated with the candidates yields a
 * distribution at every candidate position (Chapitre 9 §9.1); with a tree,
 * all branches are scored in one pass under a mask encoding the tree
 * (glossary, Medusa "Tree attention" and "L'attention en arbre"; §9.2 EAGLE-2
 * "masque personnalisé").
 *
 * For query node t of sequence b and query head h (KV head h / (Hq/Hkv)):
 *   keys allowed = prefix slots [0, L_b)  and  new-row slots L_b + j for every
 *                  node j on the root->t path;
 *   out = sum_j softmax_j(scale * q.k_j) v_j   over allowed keys.
 * Layouts: q, out [B,T,Hq,D]; k, v [B,Hkv,S_max,D]; node j's K/V row sits in
 * slot L_b + j.  bf16 inputs are raw uint16 bits.  The dense explicit mask
 * over all L_b+T keys is evaluated key by key, scores and sums in double.
 *
 * sel: optional list of nsel (b, t, h) triples; when given only those output
 * rows are computed (the rest of out is untouched), so that full-size
 * problems can be checked on a sample.
 */
int orc_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *prefix_lens, const int32_t *parents,
                       int B, int T, int Hq, int Hkv, int D, int S_max, double scale,
                       const int32_t *sel, int nsel, double *out)
{
    if (B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return ORC_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    uint8_t *mask = (uint8_t *)malloc((size_t)T * T);
    double *scores = NULL;
    int rc = ORC_OK;
    int count = sel ? nsel : B * T * Hq;
    for (int it = 0; it < count && rc == ORC_OK; ++it) {
        int b, t, h;
        if (sel) {
            b = sel[3 * it + 0];
            t = sel[3 * it + 1];
            h = sel[3 * it + 2];
        } else {
            b = it / (T * Hq);
            t = (it / Hq) % T;
            h = it % Hq;
        }
        if (b < 0 || b >= B || t < 0 || t >= T || h < 0 || h >= Hq) {
            rc = ORC_ERR_INVALID_ARG;
            break;
        }
        const int32_t *par_b = parents ? parents + (size_t)b * T : NULL;
        rc = orc_ancestor_mask(par_b, T, mask, NULL);
        if (rc != ORC_OK)
            break;
        const int L = prefix_lens[b];
        if (L < 0 || L + T > S_max) {
            rc = ORC_ERR_BAD_INPUT;
            break;
        }
        const int nkeys = L + T;
        scores = (double *)realloc(scores, sizeof(double) * (size_t)nkeys);
        const int kvh = h / G;
        const uint16_t *qrow = q + (((size_t)b * T + t) * Hq + h) * D;
        const uint16_t *kbase = k + ((size_t)b * Hkv + kvh) * (size_t)S_max * D;
        const uint16_t *vbase = v + ((size_t)b * Hkv + kvh) * (size_t)S_max * D;
        double mx = -INFINITY;
        for (int j = 0; j < nkeys; ++j) {
            int allowed = (j < L) ? 1 : mask[(size_t)t * T + (j - L)];
            if (!allowed) {
                scores[j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += bf16_bits_to_double(qrow[d]) *
                       bf16_bits_to_double(kbase[(size_t)j * D + d]);
            scores[j] = scale * acc;
            if (scores[j] > mx)
                mx = scores[j];
        }
        double z = 0.0;
        for (int j = 0; j < nkeys; ++j) {
            double w = (scores[j] == -INFINITY) ? 0.0 : exp(scores[j] - mx);
            scores[j] = w;
            z += w;
        }
        double *orow = out + (((size_t)b * T + t) * Hq + h) * D;
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j < nkeys; ++j)
                if (scores[j] != 0.0)
                    acc += scores[j] * bf16_bits_to_double(vbase[(size_t)j * D + d]);
            orow[d] = acc / z;
        }
    }
    free(scores);
    free(mask);
    return rc;
}

/* ---- A3: softmax row statistics ---------------------------------------- */

/*
 * p and q in the acceptance rule are normalised distributions (§9.1), so the
 * rule needs, per logits row: m = max_v l(v), s = sum_v exp(l(v) - m), and for
 * greedy acceptance the argmax (smallest index among equal maxima).
 */
void orc_row_stats(const void *logits, int dtype, int V, double *m_out, double *s_out,
                   int32_t *argmax_out)
{
    double m = -INFINITY;
    int32_t am = -1;
    for (int v = 0; v < V; ++v) {
        double x = logit_at(logits, dtype, (size_t)v);
        if (x > m) {
            m = x;
            am = v;
        }
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v)
        s += exp(logit_at(logits, dtype, (size_t)v) - m);
    if (m_out)
        *m_out = m;
    if (s_out)
        *s_out = s;
    if (argmax_out)
        *argmax_out = am;
}

/* probability of token v under one row: exp(l(v) - m) / s */
static double row_prob(const void *row, int dtype, int v, double m, double s)
{
    return exp(logit_at(row, dtype, (size_t)v) - m) / s;
}

/* ---- A4 + A5: stochastic chain acceptance ------------------------------ */

/*
 * Inverse-CDF draw from weights r[0..V): y = min{k : C_k > theta} with
 * C_k = r[0] + ... + r[k] summed in index order and theta = u * S.  If
 * rounding leaves no such k, the last k with r[k] > 0 is taken.  Sets
 * *near_tie when theta lies within 1e-6*S of C_{y-1} or C_y.
 */
static int32_t inverse_cdf(const double *r, int V, double S, double u, int *near_tie)
{
    const double theta = u * S;
    double c = 0.0, prev = 0.0;
    int32_t y = -1;
    for (int kk = 0; kk < V; ++kk) {
        prev = c;
        c += r[kk];
        if (c > theta) {
            y = kk;
            break;
        }
    }
    if (y < 0) {
        for (int kk = V - 1; kk >= 0; --kk)
            if (r[kk] > 0.0) {
                y = kk;
                break;
            }
        *near_tie = 1;
        return y;
    }
    const double tol = 1e-6 * S;
    if (fabs(theta - prev) < tol || fabs(theta - c) < tol)
        *near_tie = 1;
    return y;
}

/*
 * Speculative sampling on a chain (Chapitre 9 §9.1): the target produces a
 * distribution p_i at each of the N+1 positions; draft token x_i (drawn from
 * the draft's q_i) is accepted with probability min(1, p_i(x_i)/q_i(x_i)),
 * positions left to right; the first rejected position a is replaced by a
 * draw from the normalised residual (p_a - q_a)+; when all N are accepted a
 * bonus token is drawn from p_N.  Output is then distributed exactly as the
 * target alone would sample (§9.1; glossary, "Speculative Decoding (Google, 2022)").
 *
 * Readings: accept_i <=> u_accept[i] * q_i(x_i) < p_i(x_i) with u in [0,1);
 * a sequence with a draft token outside [0, V) or a logits row whose max or
 * normaliser is not finite (NaN, +inf, or every logit -inf) is invalid input;
 * one extra uniform u_sample per sequence drives the single resample / bonus
 * draw through an inverse CDF in index order; if the residual sums to zero
 * the draw falls back to p_a.  Logits arrive already temperature-scaled.
 *
 * Layouts: target [B, N+1, V], draft [B, N, V] (dtype 0 f32 / 1 bf16);
 * draft_tokens, u_accept [B, N]; u_sample [B]; accepted_len [B];
 * out_tokens [B, N+1] (x_0..x_{a-1}, then the resampled/bonus token, then -1);
 * probs [B, N, 2] = (p_i(x_i), q_i(x_i)) for every i (nullable);
 * flags [B] (ORC_FLAG_* bits, nullable); status [B] (nullable).
 */
int orc_verify_chain(const void *target, const void *draft, int dtype,
                     const int32_t *draft_tokens, const float *u_accept, const float *u_sample,
                     int B, int N, int V, int32_t *accepted_len, int32_t *out_tokens,
                     double *probs, int32_t *flags, int32_t *status)
{
    if (B <= 0 || N < 0 || V <= 0 || (dtype != 0 && dtype != 1))
        return ORC_ERR_INVALID_ARG;
    const size_t esz = dtype == 0 ? 4 : 2;
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int32_t flag = 0, st = ORC_OK;
        for (int i = 0; i <= N; ++i)
            out_tokens[(size_t)b * (N + 1) + i] = -1;
        for (int i = 0; i < N; ++i)
            if (draft_tokens[(size_t)b * N + i] < 0 || draft_tokens[(size_t)b * N + i] >= V)
                st = ORC_ERR_BAD_INPUT;
        /* a row whose max or normaliser is not finite defines no distribution */
        for (int i = 0; i < 2 * N + 1 && st == ORC_OK; ++i) {
            const char *row = i <= N
                ? (const char *)target + ((size_t)b * (N + 1) + i) * V * esz
                : (const char *)draft + ((size_t)b * N + (i - N - 1)) * V * esz;
            double m, s;
            orc_row_stats(row, dtype, V, &m, &s, NULL);
            if (!isfinite(m) || !isfinite(s) || !(s > 0.0))
                st = ORC_ERR_BAD_INPUT;
        }
        if (st != ORC_OK) {
            accepted_len[b] = -1;
            if (flags)
                flags[b] = 0;
            if (status)
                status[b] = st;
            continue;
        }
        int a = N;
        for (int i = 0; i < N; ++i) {
            const char *trow = (const char *)target + ((size_t)b * (N + 1) + i) * V * esz;
            const char *drow = (const char *)draft + ((size_t)b * N + i) * V * esz;
            double mt, st_, md, sd;
            orc_row_stats(trow, dtype, V, &mt, &st_, NULL);
            orc_row_stats(drow, dtype, V, &md, &sd, NULL);
            const int x = draft_tokens[(size_t)b * N + i];
            const double p = row_prob(trow, dtype, x, mt, st_);
            const double qq = row_prob(drow, dtype, x, md, sd);
            if (probs) {
                probs[((size_t)b * N + i) * 2 + 0] = p;
                probs[((size_t)b * N + i) * 2 + 1] = qq;
            }
            if (a < N)
                continue; /* already rejected earlier: probabilities only */
            const double uq = (double)u_accept[(size_t)b * N + i] * qq;
            if (fabs(uq - p) < 1e-6 * p)
                flag |= ORC_FLAG_ACCEPT_NEAR_TIE;
            if (!(uq < p))
                a = i;
        }
        /* the distribution the final token is drawn from */
        const char *trow = (const char *)target + ((size_t)b * (N + 1) + a) * V * esz;
        double mt, stt;
        orc_row_stats(trow, dtype, V, &mt, &stt, NULL);
        double S = 0.0;
        if (a < N) {
            const char *drow = (const char *)draft + ((size_t)b * N + a) * V * esz;
            double md, sd;
            orc_row_stats(drow, dtype, V, &md, &sd, NULL);
            for (int v = 0; v < V; ++v) {
                double diff = row_prob(trow, dtype, v, mt, stt) - row_prob(drow, dtype, v, md, sd);
                r[v] = diff > 0.0 ? diff : 0.0;
                S += r[v];
            }
            if (!(S > 0.0)) {
                flag |= ORC_FLAG_DEGENERATE_RESIDUAL;
                S = 0.0;
                for (int v = 0; v < V; ++v) {
                    r[v] = row_prob(trow, dtype, v, mt, stt);
                    S += r[v];
                }
            }
        } else {
            for (int v = 0; v < V; ++v) {
                r[v] = row_prob(trow, dtype, v, mt, stt);
                S += r[v];
            }
        }
        int near = 0;
        const int32_t y = inverse_cdf(r, V, S, (double)u_sample[b], &near);
        if (near)
            flag |= ORC_FLAG_SAMPLE_NEAR_TIE;
        for (int i = 0; i < a; ++i)
            out_tokens[(size_t)b * (N + 1) + i] = draft_tokens[(size_t)b * N + i];
        out_tokens[(size_t)b * (N + 1) + a] = y;
        accepted_len[b] = a;
        if (flags)
            flags[b] = flag;
        if (status)
            status[b] = ORC_OK;
    }
    free(r);
    return ORC_OK;
}

/* ---- A6: greedy longest agreeing path on a tree ------------------------- */

/*
 * Greedy tree acceptance (glossary "L'attention en arbre": the longest
 * accepted path becomes the generated sequence; §9.1: the longest prefix on
 * which the candidates agree with the target is kept, and at the divergence
 * the engine takes the target's own choice).
 *
 * ok[0] = 1; ok[i] = ok[parent[i]] and node_tokens[i] == argmax of the target
 * row at parent[i].  d* = the deepest ok node, the smallest index among equal
 * depths.  accepted_len = depth(d*); path_nodes = root..d*; out_tokens = the
 * tokens of path nodes 1..depth, then the target's argmax at d*.  Rows of
 * path_nodes / out_tokens are [B, T], padded with -1.
 */
int orc_verify_tree_greedy(const void *target, int dtype, const int32_t *node_tokens,
                           const int32_t *parents, int B, int T, int V,
                           int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                           int32_t *status)
{
    if (B <= 0 || T <= 0 || V <= 0 || (dtype != 0 && dtype != 1))
        return ORC_ERR_INVALID_ARG;
    const size_t esz = dtype == 0 ? 4 : 2;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    uint8_t *ok = (uint8_t *)malloc((size_t)T);
    uint8_t *mask = (uint8_t *)malloc((size_t)T * T);
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (size_t)b * T;
        const int32_t *tok = node_tokens + (size_t)b * T;
        for (int i = 0; i < T; ++i) {
            path_nodes[(size_t)b * T + i] = -1;
            out_tokens[(size_t)b * T + i] = -1;
        }
        int st = orc_ancestor_mask(par, T, mask, depth);
        for (int i = 1; i < T && st == ORC_OK; ++i)
            if (tok[i] < 0 || tok[i] >= V)
                st = ORC_ERR_BAD_INPUT;
        if (st != ORC_OK) {
            accepted_len[b] = -1;
            if (status)
                status[b] = ORC_ERR_BAD_INPUT;
            continue;
        }
        for (int i = 0; i < T; ++i) {
            const char *row = (const char *)target + ((size_t)b * T + i) * V * esz;
            orc_row_stats(row, dtype, V, NULL, NULL, &amax[i]);
        }
        ok[0] = 1;
        for (int i = 1; i < T; ++i)
            ok[i] = ok[par[i]] && tok[i] == amax[par[i]];
        int best = 0;
        for (int i = 1; i < T; ++i)
            if (ok[i] && depth[i] > depth[best])
                best = i;
        const int dd = depth[best];
        /* walk the parents from d* back to the root */
        int node = best;
        for (int d = dd; d >= 0; --d) {
            path_nodes[(size_t)b * T + d] = node;
            node = par[node];
        }
        for (int d = 1; d <= dd; ++d)
            out_tokens[(size_t)b * T + d - 1] = tok[path_nodes[(size_t)b * T + d]];
        out_tokens[(size_t)b * T + dd] = amax[best];
        accepted_len[b] = dd;
        if (status)
            status[b] = ORC_OK;
    }
    free(mask);
    free(ok);
    free(depth);
    free(amax);
    return ORC_OK;
}

/* ---- stochastic tree acceptance ------------------------------------------ */

/*
 * Multi-draft speculative sampling on a tree (the SpecInfer rule; the pages,
 * Chapitre 9 §9.2, only say that the target picks among several drafted
 * paths).  Node u's children were drawn independently from the draft's
 * distribution at u, q_u = softmax(draft row u); the target's is
 * p_u = softmax(target row u).  From the root:
 *
 *   c = 0 (the current residual is r_c = max(0, p_u - c q_u) / N(c) with
 *   N(c) = sum_v max(0, p_u(v) - c q_u(v)); c = 0 gives p_u itself);
 *   for the children v of u in index order, with token x = node_tokens[v]:
 *     accept v  <=>  u_accept[v] * q_u(x) * N(c) < max(0, p_u(x) - c q_u(x));
 *     accepted: the walk moves to v (c = 0 there);
 *     rejected: c = c + N(c).
 *   No child accepted (or u a leaf): the final token is drawn from the weights
 *   max(0, p_u - c q_u) (from p_u when they sum to zero) by the inverse CDF of
 *   inverse_cdf with u_sample.
 *
 * The update of c is the rejection step of speculative sampling applied to
 * the current residual: max(0, r_c - q_u) vanishes where p_u <= c q_u and is
 * (p_u - (c + N(c)) q_u) / N(c) elsewhere, so after normalising it is
 * r_{c + N(c)}.  It is written here in that closed form; the direct
 * recursion on vectors gives the same numbers up to rounding.
 *
 * Readings: a chain-shaped tree gives the chain rule of orc_verify_chain
 * exactly (one child per node, c = 0 at each test, c = 1 after a rejection);
 * u_accept has one uniform per node (entry 0 unused); a decision with
 * |u q N - r| < 1e-5 max(r, u q N) is a flagged near-tie (the sum N of a
 * full vocabulary differs between precisions by more than the chain's 1e-6);
 * parents, tokens and rows are checked as in the greedy walk and the chain.
 *
 * Layouts: target, draft [B, T, V] (draft row u: the distribution u's
 * children came from; leaves' rows unused); node_tokens, parents, u_accept
 * [B, T]; u_sample [B]; accepted_len [B]; path_nodes, out_tokens [B, T]
 * (-1 padded); flags, status [B] (nullable).
 */
int orc_verify_tree_stochastic(const void *target, const void *draft, int dtype,
                               const int32_t *node_tokens, const int32_t *parents,
                               const float *u_accept, const float *u_sample, int B, int T, int V,
                               int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                               int32_t *flags, int32_t *status)
{
    if (B <= 0 || T <= 0 || V <= 0 || (dtype != 0 && dtype != 1))
        return ORC_ERR_INVALID_ARG;
    const size_t esz = dtype == 0 ? 4 : 2;
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    uint8_t *mask = (uint8_t *)malloc((size_t)T * T);
    double *pu = (double *)malloc(sizeof(double) * (size_t)V);
    double *qu = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (size_t)b * T;
        const int32_t *tok = node_tokens + (size_t)b * T;
        int32_t flag = 0;
        for (int i = 0; i < T; ++i) {
            path_nodes[(size_t)b * T + i] = -1;
            out_tokens[(size_t)b * T + i] = -1;
        }
        int st = orc_ancestor_mask(par, T, mask, depth);
        for (int i = 1; i < T && st == ORC_OK; ++i)
            if (tok[i] < 0 || tok[i] >= V)
                st = ORC_ERR_BAD_INPUT;
        /* every target row, and the draft row of every node with children,
           must define a distribution */
        for (int i = 0; i < T && st == ORC_OK; ++i) {
            int has_child = 0;
            for (int j = i + 1; j < T; ++j)
                if (par[j] == i)
                    has_child = 1;
            for (int which = 0; which < 1 + has_child && st == ORC_OK; ++which) {
                const char *row = (const char *)(which ? draft : target) + ((size_t)b * T + i) * V * esz;
                double m, s;
                orc_row_stats(row, dtype, V, &m, &s, NULL);
                if (!isfinite(m) || !isfinite(s) || !(s > 0.0))
                    st = ORC_ERR_BAD_INPUT;
            }
        }
        if (st != ORC_OK) {
            accepted_len[b] = -1;
            if (flags)
                flags[b] = 0;
            if (status)
                status[b] = ORC_ERR_BAD_INPUT;
            continue;
        }
        int u = 0, dd = 0;
        path_nodes[(size_t)b * T] = 0;
        double c = 0.0;
        for (;;) {
            const char *trow = (const char *)target + ((size_t)b * T + u) * V * esz;
            const char *drow = (const char *)draft + ((size_t)b * T + u) * V * esz;
            double mt, sT, md, sd;
            orc_row_stats(trow, dtype, V, &mt, &sT, NULL);
            orc_row_stats(drow, dtype, V, &md, &sd, NULL);
            for (int v = 0; v < V; ++v) {
                pu[v] = row_prob(trow, dtype, v, mt, sT);
                qu[v] = row_prob(drow, dtype, v, md, sd);
            }
            c = 0.0;
            int next = -1;
            for (int v = u + 1; v < T && next < 0; ++v) {
                if (par[v] != u)
                    continue;
                double n = 0.0; /* N(c) */
                if (c == 0.0) {
                    n = 1.0;
                } else {
                    for (int k = 0; k < V; ++k) {
                        const double d = pu[k] - c * qu[k];
                        n += d > 0.0 ? d : 0.0;
                    }
                }
                const int x = tok[v];
                const double r = pu[x] - c * qu[x] > 0.0 ? pu[x] - c * qu[x] : 0.0;
                const double lhs = (double)u_accept[(size_t)b * T + v] * qu[x] * n;
                const double big = r > lhs ? r : lhs;
                if (fabs(lhs - r) < 1e-5 * big)
                    flag |= ORC_FLAG_ACCEPT_NEAR_TIE;
                if (lhs < r)
                    next = v;
                else
                    c += n;
            }
            if (next >= 0) {
                u = next;
                ++dd;
                path_nodes[(size_t)b * T + dd] = u;
                out_tokens[(size_t)b * T + dd - 1] = tok[u];
                continue;
            }
            /* no child accepted, or a leaf: the final draw */
            double S = 0.0;
            for (int k = 0; k < V; ++k) {
                const double d = pu[k] - c * qu[k];
                w[k] = c == 0.0 ? pu[k] : (d > 0.0 ? d : 0.0);
                S += w[k];
            }
            if (!(S > 0.0)) {
                flag |= ORC_FLAG_DEGENERATE_RESIDUAL;
                S = 0.0;
                for (int k = 0; k < V; ++k) {
                    w[k] = pu[k];
                    S += w[k];
                }
            }
            int near = 0;
            out_tokens[(size_t)b * T + dd] = inverse_cdf(w, V, S, (double)u_sample[b], &near);
            if (near)
                flag |= ORC_FLAG_SAMPLE_NEAR_TIE;
            break;
        }
        accepted_len[b] = dd;
        if (flags)
            flags[b] = flag;
        if (status)
            status[b] = ORC_OK;
    }
    free(w);
    free(qu);
    free(pu);
    free(mask);
    free(depth);
    return ORC_OK;
}

/* ---- A7: KV compaction --------------------------------------------------- */

/*
 * The enlarged KV cache holds one row per candidate node (glossary, "Limites
 * du parallel decoding").  After acceptance the accepted path's rows become
 * the committed continuation and the rest is discarded (§9.1).  Reading: node
 * j's row sits in slot L_b + j; path row d moves to slot L_b + d for
 * d = 0..a, and the cache length becomes L_b + a + 1.  path_nodes == NULL
 * means a chain (path[d] = d: nothing moves).  A path must start at the root
 * (path[0] = 0) and increase strictly, with L_b + path[d] < S_max.
 *
 * Written out of place: k_out/v_out start as copies of k_in/v_in and only the
 * destination rows are overwritten from the untouched inputs.  A sequence
 * whose accepted_len is negative (an upstream error) is left as it was.
 */
int orc_compact_kv(const uint16_t *k_in, const uint16_t *v_in, uint16_t *k_out, uint16_t *v_out,
                   const int32_t *prefix_lens, const int32_t *path_nodes,
                   const int32_t *accepted_len, int B, int Hkv, int D, int S_max,
                   int path_stride, int32_t *new_kv_lens, int32_t *status)
{
    if (B <= 0 || Hkv <= 0 || D <= 0 || S_max <= 0)
        return ORC_ERR_INVALID_ARG;
    const size_t total = (size_t)B * Hkv * S_max * D;
    memcpy(k_out, k_in, total * sizeof(uint16_t));
    memcpy(v_out, v_in, total * sizeof(uint16_t));
    for (int b = 0; b < B; ++b) {
        const int L = prefix_lens[b];
        const int a = accepted_len[b];
        int st = ORC_OK;
        if (a < 0) {
            new_kv_lens[b] = L;
            if (status)
                status[b] = ORC_OK;
            continue;
        }
        if (L < 0 || L + a + 1 > S_max || (path_nodes && a >= path_stride))
            st = ORC_ERR_BAD_INPUT;
        /* a valid path starts at the root (node 0) and increases strictly */
        for (int d = 0; d <= a && st == ORC_OK && path_nodes; ++d) {
            int src = path_nodes[(size_t)b * path_stride + d];
            if ((d == 0 && src != 0) || L + src >= S_max ||
                (d > 0 && src <= path_nodes[(size_t)b * path_stride + d - 1]))
                st = ORC_ERR_BAD_INPUT;
        }
        if (st != ORC_OK) {
            new_kv_lens[b] = L;
            if (status)
                status[b] = st;
            continue;
        }
        for (int h = 0; h < Hkv; ++h) {
            const size_t base = ((size_t)b * Hkv + h) * (size_t)S_max * D;
            for (int d = 0; d <= a; ++d) {
                const int src = path_nodes ? path_nodes[(size_t)b * path_stride + d] : d;
                memcpy(k_out + base + (size_t)(L + d) * D, k_in + base + (size_t)(L + src) * D,
                       sizeof(uint16_t) * D);
                memcpy(v_out + base + (size_t)(L + d) * D, v_in + base + (size_t)(L + src) * D,
                       sizeof(uint16_t) * D);
            }
        }
        new_kv_lens[b] = L + a + 1;
        if (status)
            status[b] = ORC_OK;
    }
    return ORC_OK;
}
