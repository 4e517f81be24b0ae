// sv_vocab.cu -- full-vocabulary passes of the verification step.
//
// Chain (stochastic) acceptance, "Chapitre 9 -- Décodage spéculatif" §9.1:
//   statistics  rows 16-byte aligned: chain_stats_stream_kernel, a persistent
//               grid (one CTA per SM, or the SMs a fused step leaves it)
//               streaming the units (sequence, row, 32 KB chunk) through a
//               ring of bulk copies; every consumer warp leaves a (max, sum
//               of exp2) record of its eighth of a unit.  Unaligned rows:
//               chain_stats_kernel, one CTA per (row, chunk), the same records.
//   decisions + draw  chain_residual_kernel: every CTA of a sequence first
//               merges the sequence's records and takes the decisions
//               u * q(x) < p(x) (p, q from an accurate exp2); then per chunk
//               of the row pair at the first rejection a it sums the weights
//               max(0, p_a - q_a) (or p_N for the bonus); the last CTA of the
//               sequence locates u * S in the chunk totals, then the thread,
//               then the element.  Whole-GPU calls with at most 16 chunks a
//               row and room for the clusters: the sequence's CTAs form a
//               cluster, the totals go through distributed shared memory,
//               and the CTA holding the crossing searches its own words.
// Greedy tree acceptance ("Parallel Decoding" glossary, "L'attention en
// arbre"; §9.1): tree_stats_stream_kernel, the same streaming pass in argmax
// mode, then tree_decide_kernel, one CTA per sequence: the rows' argmax from
// the records and the walk (every node's ancestor chain in parallel).
// Unaligned rows: tree_stats_kernel, whose last CTA per sequence walks.
// Stochastic tree acceptance (multi-draft, the SpecInfer rule): below.
//
// No CTA ever waits for another: the "last CTA" is whoever brings a
// per-sequence arrival counter to its final value; it resets the counter.
#include <climits>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

// Kernel spans (a diagnostic build only, -DSV_PHASE_STAMPS): the first start
// and the last end (globaltimer) of each streaming / decision kernel over the
// launches since sv_debug_vocab_clear, read by sv_debug_vocab_spans.  The
// library proper compiles them out.
#ifdef SV_PHASE_STAMPS
enum { kSpanChainStats, kSpanChainResidual, kSpanTreeStats, kSpanTreeDecide, kSpanCount };
static __device__ unsigned long long g_vspan[kSpanCount][2];
__device__ __forceinline__ unsigned long long span_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
struct SpanGuard {  // the end is taken at every exit of the warp
    int id;
    __device__ explicit SpanGuard(int i) : id(i) {
        if (threadIdx.x == 0) atomicMin(&g_vspan[id][0], span_now());
    }
    __device__ ~SpanGuard() {
        if ((threadIdx.x & 31) == 0) atomicMax(&g_vspan[id][1], span_now());
    }
};
#define SV_SPAN(id) SpanGuard sv_span_guard_(id)
#else
#define SV_SPAN(id) ((void)0)
#endif

constexpr int kVT = 256;                   // threads per vocabulary CTA
constexpr int kVWarps = kVT / 32;
constexpr int kLoadsPerThread = 8;         // 16-byte loads per thread per streaming item
constexpr int kResLoadsPerThread = 4;      // 16-byte loads per thread per row in the residual draw
constexpr int kMaxChainN = 63;
constexpr int kMaxTreeT = 1024;

template <typename T>
struct Elem;

template <>
struct Elem<uint16_t> {  // bf16
    static constexpr int kPerVec = 8;
    __device__ static float at(const uint16_t *p, size_t i) { return bf16_to_f32(__ldg(p + i)); }
    __device__ static void unpack(const uint4 &v, float (&x)[8]) {
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
        x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
        x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    }
};

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    __device__ static float at(const float *p, size_t i) { return __ldg(p + i); }
    __device__ static void unpack(const uint4 &v, float (&x)[4]) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
};

// ---------------------------------------------------------------- streaming chunk

// First maximum of row[begin, end) over the thread's elements and its index.
// Vector loads are laid out so that consecutive threads read consecutive
// 16-byte words; `begin` is a multiple of the vector width.
template <typename T, bool VEC>
__device__ __forceinline__ void chunk_thread_argmax(const T *row, int begin, int end,
                                                    float &best, int &idx) {
    constexpr int PV = Elem<T>::kPerVec;
    const int tid = threadIdx.x;
    best = kNegInf;
    idx = INT_MAX;
    if (VEC) {
        const int nvec = (end - begin) / PV;
        const uint4 *src = reinterpret_cast<const uint4 *>(row + begin);
        uint4 buf[kLoadsPerThread];
#pragma unroll
        for (int k = 0; k < kLoadsPerThread; ++k) {
            const int vi = k * kVT + tid;
            if (vi < nvec) buf[k] = ldg_stream(src + vi);
        }
#pragma unroll
        for (int k = 0; k < kLoadsPerThread; ++k) {
            const int vi = k * kVT + tid;
            if (vi < nvec) {
                float x[PV];
                Elem<T>::unpack(buf[k], x);
#pragma unroll
                for (int j = 0; j < PV; ++j)
                    if (x[j] > best) {
                        best = x[j];
                        idx = begin + vi * PV + j;
                    }
            }
        }
        const int tail = begin + nvec * PV + tid;  // < PV leftover elements
        if (tid < (end - begin) - nvec * PV) {
            const float xt = Elem<T>::at(row, tail);
            if (xt > best) {
                best = xt;
                idx = tail;
            }
        }
    } else {
        for (int e = begin + tid; e < end; e += kVT) {
            const float x = Elem<T>::at(row, e);
            if (x > best) {
                best = x;
                idx = e;
            }
        }
    }
}

// A 16-byte word of -inf logits: padding that contributes nothing.
template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec() {
    return sizeof(T) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                          : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Largest element of one 16-byte word (bf16: packed maxima, exact; NaN
// never wins over a number).
template <typename T>
__device__ __forceinline__ float word_max(const uint4 &v) {
    if (sizeof(T) == 2) {
        const uint32_t a = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
        return fmaxf(bf16_lo(a), bf16_hi(a));
    }
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Largest element of the thread's loaded words (bf16: packed maxima, exact).
template <typename T, int NW = kLoadsPerThread>
__device__ __forceinline__ float words_max(const uint4 (&buf)[NW]) {
    if (sizeof(T) == 2) {
        uint32_t a = bmax2(buf[0].x, buf[0].y), c = bmax2(buf[0].z, buf[0].w);
#pragma unroll
        for (int k = 1; k < NW; ++k) {
            a = bmax2(a, bmax2(buf[k].x, buf[k].y));
            c = bmax2(c, bmax2(buf[k].z, buf[k].w));
        }
        a = bmax2(a, c);
        return fmaxf(bf16_lo(a), bf16_hi(a));
    } else {
        float a = kNegInf, c = kNegInf;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            a = fmaxf(a, fmaxf(__uint_as_float(buf[k].x), __uint_as_float(buf[k].y)));
            c = fmaxf(c, fmaxf(__uint_as_float(buf[k].z), __uint_as_float(buf[k].w)));
        }
        return fmaxf(a, c);
    }
}

__device__ __forceinline__ float2 ex2_pair(float2 t) {
    return make_float2(ex2_approx(t.x), ex2_approx(t.y));
}

// Sum of exp2(x * log2 e - m) over the thread's loaded words, two elements
// per f32x2 instruction.
template <typename T, int NW = kLoadsPerThread>
__device__ __forceinline__ float words_sumexp(const uint4 (&buf)[NW], float m) {
    const float2 l2 = make_float2(kLog2e, kLog2e), nm = make_float2(-m, -m);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const uint4 v = buf[k];
        float2 x0, x1, x2, x3;
        if (sizeof(T) == 2) {
            x0 = make_float2(bf16_lo(v.x), bf16_hi(v.x));
            x1 = make_float2(bf16_lo(v.y), bf16_hi(v.y));
            x2 = make_float2(bf16_lo(v.z), bf16_hi(v.z));
            x3 = make_float2(bf16_lo(v.w), bf16_hi(v.w));
            acc0 = __fadd2_rn(acc0, ex2_pair(__ffma2_rn(x0, l2, nm)));
            acc1 = __fadd2_rn(acc1, ex2_pair(__ffma2_rn(x1, l2, nm)));
            acc0 = __fadd2_rn(acc0, ex2_pair(__ffma2_rn(x2, l2, nm)));
            acc1 = __fadd2_rn(acc1, ex2_pair(__ffma2_rn(x3, l2, nm)));
        } else {
            x0 = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
            x1 = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
            acc0 = __fadd2_rn(acc0, ex2_pair(__ffma2_rn(x0, l2, nm)));
            acc1 = __fadd2_rn(acc1, ex2_pair(__ffma2_rn(x1, l2, nm)));
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// Statistics of row[begin, end) over the whole CTA: the chunk's maximum
// first (scaled by log2 e into m), then every thread sums exp2 against that
// one maximum, so the sums add without rescaling.  (m, s) valid in thread 0.
template <typename T, bool VEC>
__device__ __forceinline__ void chunk_cta_stats(const T *row, int begin, int end,
                                                float *red /* [2 * kVWarps] */, float &m_out,
                                                float &s_out) {
    constexpr int PV = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint4 buf[kLoadsPerThread];
    float xt = kNegInf;
    float vmax = kNegInf;
    if (VEC) {
        const int nvec = (end - begin) / PV;
        const uint4 *src = reinterpret_cast<const uint4 *>(row + begin);
#pragma unroll
        for (int k = 0; k < kLoadsPerThread; ++k) {
            const int vi = k * kVT + tid;
            buf[k] = vi < nvec ? ldg_stream(src + vi) : neg_inf_vec<T>();
        }
        const int tail = begin + nvec * PV + tid;  // < PV leftover elements
        if (tid < (end - begin) - nvec * PV) xt = Elem<T>::at(row, tail);
        vmax = fmaxf(words_max<T>(buf), xt);
    } else {
        for (int e = begin + tid; e < end; e += kVT) vmax = fmaxf(vmax, Elem<T>::at(row, e));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    if (lane == 0) red[warp] = vmax;
    __syncthreads();
    float cmax = red[0];
#pragma unroll
    for (int w = 1; w < kVWarps; ++w) cmax = fmaxf(cmax, red[w]);
    const float m = cmax * kLog2e;
    float s = 0.f;
    if (m != kNegInf) {  // the same decision in every thread
        if (VEC) {
            s = words_sumexp<T>(buf, m);
            if (xt != kNegInf) s += ex2_approx(fmaf(xt, kLog2e, -m));
        } else {
            for (int e = begin + tid; e < end; e += kVT)
                s += ex2_approx(fmaf(Elem<T>::at(row, e), kLog2e, -m));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) red[kVWarps + warp] = s;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kVWarps; ++w) t += red[kVWarps + w];
        m_out = m;
        s_out = t;
    }
}

// Reduce per-thread statistics over the CTA; the result is valid in thread 0.
template <bool ARGMAX>
__device__ __forceinline__ void cta_reduce_stats(float &m, float &s, float &best, int &idx,
                                                 float4 *scratch /* [kVWarps] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (ARGMAX) {
            const float b2 = __shfl_xor_sync(0xffffffffu, best, off);
            const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
            merge_argmax(best, idx, b2, i2);
        } else {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            merge_ms(m, s, m2, s2);
        }
    }
    if (lane == 0) scratch[warp] = make_float4(m, s, best, __int_as_float(idx));
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kVWarps; ++w) {
            const float4 o = scratch[w];
            if (ARGMAX)
                merge_argmax(best, idx, o.z, __float_as_int(o.w));
            else
                merge_ms(m, s, o.x, o.y);
        }
    }
}

// Merge the chunk partials of one row, one warp; result valid in lane 0.
template <bool ARGMAX>
__device__ __forceinline__ RowPartial warp_merge_row(const RowPartial *parts, int nchunks) {
    const int lane = threadIdx.x & 31;
    float m = kNegInf, s = 0.f, best = kNegInf;
    int idx = INT_MAX;
    for (int c = lane; c < nchunks; c += 32) {
        const float4 p = __ldcg(reinterpret_cast<const float4 *>(parts + c));
        if (ARGMAX)
            merge_argmax(best, idx, p.z, __float_as_int(p.w));
        else
            merge_ms(m, s, p.x, p.y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (ARGMAX) {
            const float b2 = __shfl_xor_sync(0xffffffffu, best, off);
            const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
            merge_argmax(best, idx, b2, i2);
        } else {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            merge_ms(m, s, m2, s2);
        }
    }
    RowPartial r;
    r.m = m;
    r.s = s;
    r.best = best;
    r.idx = idx;
    return r;
}

struct WsView {
    int *counters;  // [B] tree pass, [B] residual draw, [1] statistics pass timed out
    RowPartial *partials;
    float2 *chunktot;
};

__host__ __device__ inline WsView ws_view(void *ws, const VocabPlan &p, int B) {
    char *base = static_cast<char *>(ws);
    WsView v;
    v.counters = reinterpret_cast<int *>(base + p.off_counters);
    v.partials = reinterpret_cast<RowPartial *>(base + p.off_partials);
    v.chunktot = reinterpret_cast<float2 *>(base + p.off_chunktot);
    (void)B;
    return v;
}

// ---------------------------------------------------------------- chain: kernel 1

// Draft length N_b of chain sequence b (N without a length array; 0 for an
// invalid length, whose sequence the decisions report).
__device__ __forceinline__ int chain_draft_len(const ChainArgs &a, int b) {
    if (!a.draft_lens) return a.N;
    const int n = a.draft_lens[b];
    return (n >= 0 && n <= a.N) ? n : 0;
}

// Row r of the [target rows 0..N, draft rows 0..N-1] order is in use for a
// sequence with N_b drafts: target rows 0..N_b and draft rows 0..N_b-1.  The
// others are padding, never read.
__device__ __forceinline__ bool chain_row_in_use(int N, int nb, int r) {
    return r <= nb || (r > N && r - N - 1 < nb);
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kVT, 5) chain_stats_kernel(ChainArgs a, VocabPlan p, WsView w) {
    __shared__ float red[2 * kVWarps];
    const int R = 2 * a.N + 1;
    const int per_seq = R * p.nchunks;
    const int item = blockIdx.x;
    const int b = item / per_seq;
    const int rem = item - b * per_seq;
    const int r = rem / p.nchunks;
    const int c = rem - r * p.nchunks;
    const T *row = r <= a.N
                       ? static_cast<const T *>(a.target) + ((size_t)b * (a.N + 1) + r) * a.V
                       : static_cast<const T *>(a.draft) + ((size_t)b * a.N + (r - a.N - 1)) * a.V;
    const int begin = c * p.chunk_elems;
    const int end = min(a.V, begin + p.chunk_elems);

    griddep_wait();
    griddep_launch_dependents();
    if (!chain_row_in_use(a.N, chain_draft_len(a, b), r)) {  // a padding row: an empty record
        if (threadIdx.x == 0) reinterpret_cast<float2 *>(w.partials)[item] = make_float2(kNegInf, 0.f);
        return;
    }
    float m = 0.f, s = 0.f;
    chunk_cta_stats<T, VEC>(row, begin, end, red, m, s);
    if (threadIdx.x == 0) reinterpret_cast<float2 *>(w.partials)[item] = make_float2(m, s);
}

// ---------------------------------------------------------------- chain: kernel 1, streaming form

// Rows 16-byte aligned (V * element size a multiple of 16): a persistent grid
// (one CTA per SM) streams the units (sequence, row, 32 KB chunk) of a
// balanced contiguous range through a ring of shared-memory stages filled by
// 1-D bulk copies (one producer thread), so the loads never wait for the
// arithmetic.  Two groups of 8 consumer warps take alternate units; each warp
// reduces an eighth of its unit on its own -- its maximum first (packed bf16
// maxima), then the sum of exp2 against it -- and leaves one (max, sum)
// record; no CTA-wide barrier.  The decisions are taken by the next kernel.
constexpr int kSWarps = 16;                      // consumer warps
constexpr int kSThreads = 32 * (kSWarps + 1);    // + the producer warp
constexpr int kSUnitBytes = 32768;               // one unit = one chunk of a row
constexpr int kSStages = 6;
constexpr int kSGroupWarps = kSWarps / 2;        // warps sharing one unit
constexpr int kSWordsPerLane = kSUnitBytes / 16 / kSGroupWarps / 32;  // 16-byte words: 8

template <typename T>
__global__ void __launch_bounds__(kSThreads, 1)
    chain_stats_stream_kernel(ChainArgs a, VocabPlan p, WsView w) {
    SV_SPAN(kSpanChainStats);
    extern __shared__ __align__(128) uint8_t ring[];  // kSStages * kSUnitBytes
    __shared__ uint64_t full[kSStages], empty[kSStages];
    constexpr int PV = Elem<T>::kPerVec;
    constexpr int kUnitElems = kSUnitBytes / (int)sizeof(T);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = 2 * a.N + 1;
    const int per_seq = R * p.nchunks;
    const long long U = (long long)a.B * per_seq;
    const long long u_begin = U * blockIdx.x / gridDim.x, u_end = U * (blockIdx.x + 1) / gridDim.x;
    float2 *rec = reinterpret_cast<float2 *>(w.partials);  // [B][R][nchunks][kSGroupWarps]

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSGroupWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    if (warp == kSWarps) {
        // ================= producer: one bulk copy per unit (evict-first: the
        // stream does not push the records and code of what follows out of L2)
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            long long k = 0;
            int cb = -1, nb = 0;  // the sequence of the last unit and its draft length
            for (long long u = u_begin; u < u_end; ++u, ++k) {
                const int s = (int)(k % kSStages);
                if (!mbar_wait_bounded(&empty[s], (uint32_t)(((k / kSStages) & 1) ^ 1))) {
                    atomicExch(w.counters + 2 * a.B, 1);  // a stage never came free
                    break;
                }
                const int b = (int)(u / per_seq);
                const int rem = (int)(u - (long long)b * per_seq);
                const int r = rem / p.nchunks, c = rem - r * p.nchunks;
                if (b != cb) {
                    cb = b;
                    nb = chain_draft_len(a, b);
                }
                if (!chain_row_in_use(a.N, nb, r)) {  // padding: the stage's phase, no copy
                    mbar_arrive(&full[s]);
                    continue;
                }
                const T *row = r <= a.N
                    ? static_cast<const T *>(a.target) + ((size_t)b * (a.N + 1) + r) * a.V
                    : static_cast<const T *>(a.draft) + ((size_t)b * a.N + (r - a.N - 1)) * a.V;
                const int begin = c * kUnitElems;
                const uint32_t bytes = (uint32_t)(min(kUnitElems, a.V - begin) * (int)sizeof(T));
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_load_hint(ring + s * kSUnitBytes, row + begin, bytes, &full[s], pol);
            }
            // every copy issued must land before the CTA may exit
            const long long first = k > kSStages ? k - kSStages : 0;
            for (long long j = first; j < k; ++j)
                mbar_wait_bounded(&full[j % kSStages], (uint32_t)((j / kSStages) & 1));
        }
        return;
    }

    // ================= consumers
    // Two groups of eight warps (one pair per SM sub-partition) take
    // alternate units, so the groups drift out of step and one group's
    // exponentials overlap the other's loads and shuffles.
    // group of warp w: (w / 4) % 2, so each sub-partition (w % 4) holds two
    // warps of each group; warp within the group: 0..7
    const int grp = (warp >> 2) & 1, gw = ((warp >> 3) << 2) | (warp & 3);
    int cb = -1, nb = 0;
    for (long long k = grp; k < u_end - u_begin; k += 2) {
        const long long u = u_begin + k;
        const int s = (int)(k % kSStages);
        const int b = (int)(u / per_seq);
        const int rem = (int)(u - (long long)b * per_seq);
        const int r = rem / p.nchunks, c = rem - r * p.nchunks;
        const int n = min(kUnitElems, a.V - c * kUnitElems);  // elements in this unit (a multiple of PV)
        if (b != cb) {
            cb = b;
            nb = chain_draft_len(a, b);
        }
        if (!warp_wait_bounded(&full[s], (uint32_t)((k / kSStages) & 1))) {
            // the record stays unwritten: the decisions report every sequence
            if (lane == 0) atomicExch(w.counters + 2 * a.B, 1);
            break;
        }
        if (!chain_row_in_use(a.N, nb, r)) {  // padding: nothing landed, an empty record
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                rec[(((size_t)b * R + r) * p.nchunks + c) * kSGroupWarps + gw] =
                    make_float2(kNegInf, 0.f);
            }
            continue;
        }
        uint4 buf[kSWordsPerLane];
#pragma unroll
        for (int q = 0; q < kSWordsPerLane; ++q) {
            const int wi = (gw * kSWordsPerLane + q) * 32 + lane;  // 16-byte word of the unit
            buf[q] = wi * PV < n ? *reinterpret_cast<const uint4 *>(ring + s * kSUnitBytes + wi * 16)
                                 : neg_inf_vec<T>();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the words are in registers
        // the warp's maximum first, then every lane sums exp2 against it
        // (no exponentials spent on merging lanes)
        float vmax = words_max<T, kSWordsPerLane>(buf);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        const float m = vmax * kLog2e;
        float sum = m == kNegInf ? 0.f : words_sumexp<T, kSWordsPerLane>(buf, m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0)
            rec[(((size_t)b * R + r) * p.nchunks + c) * kSGroupWarps + gw] = make_float2(m, sum);
    }
}

// ---------------------------------------------------------------- chain: kernel 2

// Weights of the residual draw.  mode 0: r = max(0, p - q); mode 1: r = p.
// Written with explicitly rounded operations so that recomputing a weight
// gives identical bits.
template <typename T>
struct ResidualRow {
    const T *trow;
    const T *drow;
    float ms_t, inv_t, ms_d, inv_d;

    __device__ __forceinline__ float p_at(float lt) const {
        return __fmul_rn(ex2_approx(__fmaf_rn(lt, kLog2e, -ms_t)), inv_t);
    }
    __device__ __forceinline__ float q_at(float ld) const {
        return __fmul_rn(ex2_approx(__fmaf_rn(ld, kLog2e, -ms_d)), inv_d);
    }
};

// Raw 32-bit word `bits` of element i (bf16: zero-extended half).
template <typename T>
__device__ __forceinline__ uint32_t elem_bits(const T *row, int i) {
    if (sizeof(T) == 2) return __ldg(reinterpret_cast<const unsigned short *>(row) + i);
    return __float_as_uint(__ldg(reinterpret_cast<const float *>(row) + i));
}

// The thread's elements [e0, e0 + n) of one row as raw 16-byte words;
// elements at and past n read as -inf (weight 0).
template <typename T, bool VEC>
__device__ __forceinline__ void load_res_words(const T *row, int e0, int n,
                                               uint4 (&raw)[kResLoadsPerThread]) {
    constexpr int PV = Elem<T>::kPerVec;
    if (VEC && n == kResLoadsPerThread * PV) {
        const uint4 *src = reinterpret_cast<const uint4 *>(row + e0);
#pragma unroll
        for (int k = 0; k < kResLoadsPerThread; ++k) raw[k] = __ldg(src + k);
        return;
    }
#pragma unroll
    for (int k = 0; k < kResLoadsPerThread; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (sizeof(T) == 2) {
                const int j = k * PV + 2 * c;
                const uint32_t lo = j < n ? elem_bits(row, e0 + j) : 0xff80u;
                const uint32_t hi = j + 1 < n ? elem_bits(row, e0 + j + 1) : 0xff80u;
                w[c] = lo | (hi << 16);
            } else {
                const int j = k * PV + c;
                w[c] = j < n ? elem_bits(row, e0 + j) : 0xff800000u;
            }
        }
        raw[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Element j of the raw words (j a compile-time constant after unrolling).
template <typename T>
__device__ __forceinline__ float raw_elem(const uint4 (&raw)[kResLoadsPerThread], int j) {
    constexpr int PV = Elem<T>::kPerVec;
    const uint4 &v = raw[j / PV];
    const int c = sizeof(T) == 2 ? (j % PV) / 2 : j % PV;
    const uint32_t w = c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
    if (sizeof(T) == 2) return (j & 1) ? bf16_hi(w) : bf16_lo(w);
    return __uint_as_float(w);
}

template <typename T>
__device__ __forceinline__ float raw_weight(const ResidualRow<T> &rw, int mode,
                                            const uint4 (&rt)[kResLoadsPerThread],
                                            const uint4 (&rd)[kResLoadsPerThread], int j) {
    const float pj = rw.p_at(raw_elem<T>(rt, j));
    if (mode) return pj;
    return fmaxf(__fsub_rn(pj, rw.q_at(raw_elem<T>(rd, j))), 0.f);
}

// The same weight from one target logit and one draft logit.
template <typename T>
__device__ __forceinline__ float elem_weight(const ResidualRow<T> &rw, int mode, float lt, float ld) {
    const float pj = rw.p_at(lt);
    if (mode) return pj;
    return fmaxf(__fsub_rn(pj, rw.q_at(ld)), 0.f);
}

// Element j of a thread's run kept as raw 16-byte words in shared memory.
template <typename T>
__device__ __forceinline__ float smem_elem(const uint4 *words, int j) {
    if (sizeof(T) == 2)
        return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short *>(words)[j] << 16);
    return reinterpret_cast<const float *>(words)[j];
}

// Sequential sums over the thread's elements: sr of the weights in `mode`,
// sp of p (the fallback weights).
template <typename T>
__device__ __forceinline__ void raw_weight_sums(const ResidualRow<T> &rw, int mode,
                                                const uint4 (&rt)[kResLoadsPerThread],
                                                const uint4 (&rd)[kResLoadsPerThread], float &sr,
                                                float &sp) {
    constexpr int EPT = kResLoadsPerThread * Elem<T>::kPerVec;
    sr = 0.f;
    sp = 0.f;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const float pj = rw.p_at(raw_elem<T>(rt, j));
        const float wj = mode ? pj : fmaxf(__fsub_rn(pj, rw.q_at(raw_elem<T>(rd, j))), 0.f);
        sr = __fadd_rn(sr, wj);
        sp = __fadd_rn(sp, pj);
    }
}

// Inclusive prefix over the CTA's 256 per-thread pairs with a fixed order of
// additions (warp shuffle scan, then warp totals added in warp order), both
// components independently; `total` gets the sums of all 256, bitwise equal
// to thread 255's result.
__device__ __forceinline__ float2 cta_incl_scan2(float2 v, float2 &total, float2 *wsum /* [8] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float tx = __shfl_up_sync(0xffffffffu, v.x, off);
        const float ty = __shfl_up_sync(0xffffffffu, v.y, off);
        if (lane >= off) {
            v.x = __fadd_rn(v.x, tx);
            v.y = __fadd_rn(v.y, ty);
        }
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    float2 base = make_float2(0.f, 0.f), tot = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kVWarps; ++w) {
        if (w == warp) base = tot;
        tot.x = __fadd_rn(tot.x, wsum[w].x);
        tot.y = __fadd_rn(tot.y, wsum[w].y);
    }
    __syncthreads();
    total = tot;
    return warp == 0 ? v : make_float2(__fadd_rn(base.x, v.x), __fadd_rn(base.y, v.y));
}

// 2^(l * log2 e - m) in single precision to about 2e-7 relative: l * log2 e
// is carried as an exact float pair (log2 e split into a float and its
// remainder), the difference with m by an error-free two-sum, the integer
// part of the exponent applied by ldexp and the fraction f in [-1/2, 1/2]
// by the degree-7 Taylor polynomial of e^(f ln 2) (remainder below 6e-9).
__device__ __forceinline__ float exp2_diff_accurate(float l, float m) {
    constexpr float kL2eHi = 1.4426950216293335f;   // float nearest log2 e
    constexpr float kL2eLo = 1.925963033500011e-08f;  // log2 e - kL2eHi
    constexpr float kLn2 = 0.6931471824645996f;
    const float hi = l * kL2eHi;
    const float lo = __fmaf_rn(l, kL2eHi, -hi) + l * kL2eLo;  // l * log2 e = hi + lo
    const float s = __fsub_rn(hi, m);                           // two-sum of hi and -m
    const float bp = __fsub_rn(s, hi);
    const float err = __fsub_rn(hi, __fsub_rn(s, bp)) + __fsub_rn(-m, bp);
    const float n = rintf(s);
    const float f = __fsub_rn(s, n) + (err + lo);  // exponent = n + f
    const float x = f * kLn2;
    float e = 1.f + x * (1.f / 7.f);
    e = 1.f + x * (1.f / 6.f) * e;
    e = 1.f + x * (1.f / 5.f) * e;
    e = 1.f + x * (1.f / 4.f) * e;
    e = 1.f + x * (1.f / 3.f) * e;
    e = 1.f + x * (1.f / 2.f) * e;
    e = 1.f + x * e;  // e^x = 1 + x (1 + x/2 (1 + x/3 (...)))
    return ldexpf(e, (int)n);
}

// The inputs of sequence b's decisions that this thread needs (p_i's token
// and logit on threads 0..N-1, q_i's on threads 64..64+N-1, u_i on thread
// i), read before the statistics pass has finished: they are inputs of the
// call, complete once that pass let this kernel launch.
struct ChainPosIn {
    int nb_raw;   // the draft length as given
    bool tok_ok;  // the thread's token is in [0, V)
    float l;      // the logit at the token
    float u;      // u_accept of position threadIdx.x
};

template <typename T>
__device__ __forceinline__ ChainPosIn chain_pos_inputs(const ChainArgs &a, int b) {
    const int tid = threadIdx.x;
    ChainPosIn in;
    in.nb_raw = a.draft_lens ? a.draft_lens[b] : a.N;
    const int Nb = (in.nb_raw >= 0 && in.nb_raw <= a.N) ? in.nb_raw : 0;
    const int i = tid & 63;
    const int is_q = (tid >> 6) & 1;
    in.tok_ok = false;
    in.l = 0.f;
    in.u = tid < a.N ? a.u_accept[(size_t)b * a.N + tid] : 0.f;
    if (tid < 128 && i < Nb) {
        const int x = a.tokens[(size_t)b * a.N + i];
        in.tok_ok = x >= 0 && x < a.V;
        if (in.tok_ok) {
            const T *row = is_q ? static_cast<const T *>(a.draft) + ((size_t)b * a.N + i) * a.V
                                : static_cast<const T *>(a.target) + ((size_t)b * (a.N + 1) + i) * a.V;
            in.l = Elem<T>::at(row, x);
        }
    }
    return in;
}

// Decisions of sequence b from its rows' (max, sum) records, by a whole CTA:
// a warp per row merges the row's records (their maximum first, then the sums
// rescaled to it, 64 records at a time); p_i(x_i) and q_i(x_i) from the row
// statistics by exp2_diff_accurate (p and q on separate threads); accept while
// u_i * q < p; a = the first
// rejection (N if none, -1 if the sequence is invalid).  With `outputs` it
// also writes accepted_len, seq_status, probs and the emitted tokens except
// the one drawn at position a.
__device__ __forceinline__ ChainDecision decide_sequence(const ChainArgs &a, const VocabPlan &p,
                                                         const float2 *rec, const int *timed_out,
                                                         int b, bool outputs, const ChainPosIn &in) {
    __shared__ float s_ms[2 * kMaxChainN + 1][2];
    __shared__ float s_pq[kMaxChainN][2];
    __shared__ int s_bad, s_first;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = 2 * a.N + 1;
    const int per_row = p.nchunks * p.recs_per_unit;
    // this sequence's draft length; rows and positions past it are padding
    const int nb_raw = in.nb_raw;
    const bool nb_ok = nb_raw >= 0 && nb_raw <= a.N;
    const int Nb = nb_ok ? nb_raw : 0;
    if (tid == 0) {
        // bit 0: invalid input; bit 1: the statistics pass gave up (records
        // left unwritten), so no decision is taken
        s_bad = (nb_ok ? 0 : 1) | (__ldcg(timed_out) != 0 ? 2 : 0);
        s_first = Nb;
    }
    // p_i on threads 0..N-1, q_i on threads 64..64+N-1 (token and logit
    // fetched by the caller)
    const int i = tid & 63;
    const int is_q = (tid >> 6) & 1;
    const bool pos_thread = tid < 128 && i < Nb;
    const float l = in.l;
    const bool tok_ok = in.tok_ok;
    // rows: a warp per row, four rows of a warp in flight at a time; each row
    // merges its records once (their maximum, then the rescaled sums)
    for (int r0 = warp; r0 < R; r0 += 4 * kVWarps) {
        float mx[4], sm[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mx[q] = kNegInf;
            sm[q] = 0.f;
        }
        for (int i0 = 0; i0 < per_row; i0 += 64) {
            float2 v[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = r0 + q * kVWarps;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int ii = i0 + lane + 32 * j;
                    v[q][j] = (rr < R && ii < per_row)
                                  ? __ldcg(rec + ((size_t)b * R + rr) * per_row + ii)
                                  : make_float2(kNegInf, 0.f);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float cm = fmaxf(v[q][0].x, v[q][1].x);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
                float cs = 0.f;
                if (cm != kNegInf) {
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        if (v[q][j].x != kNegInf) cs += v[q][j].y * exp2f(v[q][j].x - cm);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
                merge_ms(mx[q], sm[q], cm, cs);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = r0 + q * kVWarps;
                if (rr < R) {
                    s_ms[rr][0] = mx[q];
                    s_ms[rr][1] = sm[q];
                }
            }
        }
    }
    __syncthreads();
    if (tid < R && (tid <= Nb || (tid > a.N && tid - a.N - 1 < Nb))) {  // rows in use
        const float mm = s_ms[tid][0], ss = s_ms[tid][1];
        if (!(isfinite(mm) && isfinite(ss) && ss > 0.f)) atomicOr(&s_bad, 1);
    }
    if (pos_thread) {
        float v = 0.f;
        if (!tok_ok) {
            atomicOr(&s_bad, 1);
        } else {
            const int ri = is_q ? a.N + 1 + i : i;
            v = __fdiv_rn(exp2_diff_accurate(l, s_ms[ri][0]), s_ms[ri][1]);
        }
        s_pq[i][is_q] = v;
    }
    __syncthreads();
    if (tid < a.N) {
        const bool used = tid < Nb;
        const float pp = used ? s_pq[tid][0] : 0.f, qq = used ? s_pq[tid][1] : 0.f;
        if (used && !(in.u * qq < pp)) atomicMin(&s_first, tid);
        if (outputs && a.probs) {
            a.probs[((size_t)b * a.N + tid) * 2 + 0] = pp;
            a.probs[((size_t)b * a.N + tid) * 2 + 1] = qq;
        }
    }
    __syncthreads();
    const bool late = (s_bad & 2) != 0;
    const bool bad = s_bad != 0;
    const int acc = bad ? -1 : s_first;
    ChainDecision d;
    d.n_draft = Nb;
    d.pad2[0] = d.pad2[1] = 0.f;
    d.a = acc;
    d.ms_t = bad ? 0.f : s_ms[acc][0];
    d.s_t = bad ? 0.f : s_ms[acc][1];
    d.ms_d = (!bad && acc < Nb) ? s_ms[a.N + 1 + acc][0] : 0.f;
    d.s_d = (!bad && acc < Nb) ? s_ms[a.N + 1 + acc][1] : 0.f;
    if (outputs) {
        if (tid == 0) {
            a.accepted_len[b] = acc;
            if (a.seq_status) a.seq_status[b] = late ? SV_ERR_TIMEOUT : bad ? SV_ERR_BAD_INPUT : SV_OK;
            if (a.new_kv_lens) {
                // fused step: a chain's accepted rows are already in place
                // (node d at slot L + d), so compaction is the new length
                const int L = a.prefix_lens[b];
                const bool fits = L >= 0 && (long long)L + Nb + 1 <= a.S_max;
                a.new_kv_lens[b] = (fits && acc >= 0) ? L + acc + 1 : L;
            }
        }
        for (int j = tid; j <= a.N; j += kVT) {
            int v = -1;
            if (acc >= 0 && j < acc) v = a.tokens[(size_t)b * a.N + j];
            if (acc < 0 || j != acc) a.out_tokens[(size_t)b * (a.N + 1) + j] = v;
        }
    }
    return d;
}

// CLUSTER: the CTAs of a sequence form one thread-block cluster (at most
// kMaxResCluster chunks a row); each sends its chunk totals into every
// other's shared memory, and after one cluster barrier all of them run the
// same search over the totals: the CTA whose chunk holds the crossing goes
// on with the words still in its registers, the others leave.  Otherwise
// the totals go through memory and the last CTA of the sequence to count
// its chunk searches them and loads the crossing chunk again.
template <typename T, bool VEC, bool CLUSTER>
// (Aligned rows: at most 64 registers, so that four CTAs per SM keep a
// B = 32, V = 128256 grid in one wave.)
__global__ void __launch_bounds__(kVT, VEC ? 4 : 1) chain_residual_kernel(ChainArgs a, VocabPlan p, WsView w) {
    SV_SPAN(kSpanChainResidual);
    constexpr int EPT = kResLoadsPerThread * Elem<T>::kPerVec;
    __shared__ float2 wsum[kVWarps];
    __shared__ float2 s_tot[kMaxResChunks];
    __shared__ float s_prefix[kVT];
    __shared__ int s_last, s_cstar, s_mode, s_fallback, s_pick_min, s_pick_max;
    __shared__ uint4 s_words[2][kResLoadsPerThread];  // the picked thread's run
    __shared__ float s_base, s_theta;
    // cluster form: every CTA of the cluster has started before any writes
    // into another's shared memory (the matching wait precedes the sends)
    if constexpr (CLUSTER) cluster_arrive_relaxed();

    const int b = blockIdx.x / p.res_chunks;
    const int c = blockIdx.x - b * p.res_chunks;
    // the call's inputs first, while the statistics pass may still run
    const float u_s = threadIdx.x == 0 ? a.u_sample[b] : 0.f;  // for the last CTA's search
    const ChainPosIn pin = chain_pos_inputs<T>(a, b);
    griddep_wait();
    griddep_launch_dependents();
    // every CTA of the sequence takes the decisions; the first one writes them
    const ChainDecision d =
        decide_sequence(a, p, reinterpret_cast<const float2 *>(w.partials),
                        w.counters + 2 * a.B, b, c == 0, pin);
    if (d.a < 0) return;  // invalid sequence: -1s written above

    ResidualRow<T> rw;
    rw.trow = static_cast<const T *>(a.target) + ((size_t)b * (a.N + 1) + d.a) * a.V;
    rw.drow = d.a < d.n_draft ? static_cast<const T *>(a.draft) + ((size_t)b * a.N + d.a) * a.V
                        : rw.trow;
    rw.ms_t = d.ms_t;
    rw.inv_t = __frcp_rn(d.s_t);
    rw.ms_d = d.ms_d;
    rw.inv_d = d.a < d.n_draft ? __frcp_rn(d.s_d) : 0.f;
    const int mode0 = d.a < d.n_draft ? 0 : 1;  // residual at a rejection, else the bonus

    // ---- every CTA: weight sums of its chunk (the residual's and p's)
    const int e0 = c * p.res_chunk_elems + threadIdx.x * EPT;
    const int n = max(0, min(EPT, a.V - e0));
    uint4 rt[kResLoadsPerThread], rd[kResLoadsPerThread];
    load_res_words<T, VEC>(rw.trow, e0, n, rt);
    if (mode0 == 0) load_res_words<T, VEC>(rw.drow, e0, n, rd);
    float sr, sp;
    raw_weight_sums<T>(rw, mode0, rt, rd, sr, sp);
    float2 tot;
    float2 incl = cta_incl_scan2(make_float2(sr, sp), tot, wsum);
    if constexpr (CLUSTER) {
        // this chunk's totals into slot c of every CTA of the cluster (rank
        // r = chunk r); the barrier makes them visible, and no CTA reads
        // another's shared memory after it, so any may then leave
        cluster_wait();
        if ((int)threadIdx.x < p.res_chunks)
            st_cluster_f2(cluster_map(smem_u32(&s_tot[c]), threadIdx.x), tot);
        __syncwarp();
        cluster_sync();
        (void)s_last;
    } else {
        if (threadIdx.x == 0) {
            w.chunktot[(size_t)b * p.res_chunks + c] = tot;
            __threadfence();
            const int old = atomicAdd(&w.counters[a.B + b], 1);
            s_last = (old == p.res_chunks - 1);
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();

        // ---- last CTA of sequence b: locate u * S in the chunk prefix
        for (int i = threadIdx.x; i < p.res_chunks; i += kVT)
            s_tot[i] = __ldcg(w.chunktot + (size_t)b * p.res_chunks + i);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        float S = 0.f;
        for (int i = 0; i < p.res_chunks; ++i) S = __fadd_rn(S, s_tot[i].x);
        int mode = mode0;
        if (!(S > 0.f)) {  // residual vanished: draw from p_a instead
            mode = 1;
            S = 0.f;
            for (int i = 0; i < p.res_chunks; ++i) S = __fadd_rn(S, s_tot[i].y);
        }
        const float theta = __fmul_rn(u_s, S);
        float base = 0.f;
        int cstar = -1;
        for (int i = 0; i < p.res_chunks; ++i) {
            const float t = mode == 0 ? s_tot[i].x : s_tot[i].y;
            const float nb = __fadd_rn(base, t);
            if (nb > theta) {
                cstar = i;
                break;
            }
            base = nb;
        }
        int fallback = 0;
        if (cstar < 0) {  // rounding left no crossing: last chunk with weight
            fallback = 1;
            cstar = 0;
            for (int i = p.res_chunks - 1; i >= 0; --i)
                if ((mode == 0 ? s_tot[i].x : s_tot[i].y) > 0.f) {
                    cstar = i;
                    break;
                }
        }
        s_cstar = cstar;
        s_mode = mode;
        s_fallback = fallback;
        s_base = base;
        s_theta = theta;
        s_pick_min = kVT;
        s_pick_max = -1;
    }
    __syncthreads();
    const int cstar = s_cstar, mode = s_mode;
    if (CLUSTER && cstar != c) return;  // the crossing is in another CTA's chunk
    const float base = s_base, theta = s_theta;
    const int f0 = cstar * p.res_chunk_elems + threadIdx.x * EPT;
    const int fn = max(0, min(EPT, a.V - f0));
    // ---- then chunk cstar again: its words (from L2) and the same thread
    // sums and scan as its CTA computed, so its thread prefixes need no
    // round trip through memory (the last CTA's own chunk is at hand) ...
    if (cstar != c) {
        load_res_words<T, VEC>(rw.trow, f0, fn, rt);
        if (mode0 == 0) load_res_words<T, VEC>(rw.drow, f0, fn, rd);
        raw_weight_sums<T>(rw, mode0, rt, rd, sr, sp);
        incl = cta_incl_scan2(make_float2(sr, sp), tot, wsum);
    }
    // ... the thread where the prefix passes u * S (or, after a fallback, the
    // last thread holding any weight), one vote per warp
    const float incl_m = mode == 0 ? incl.x : incl.y;
    s_prefix[threadIdx.x] = incl_m;
    const bool fb = s_fallback != 0;
    const bool hit = fb ? (mode == 0 ? sr : sp) > 0.f : __fadd_rn(base, incl_m) > theta;
    const unsigned vote = __ballot_sync(0xffffffffu, hit);
    if ((threadIdx.x & 31) == 0 && vote != 0u) {
        const int wbase = threadIdx.x & ~31;
        if (fb) atomicMax(&s_pick_max, wbase + 31 - __clz((int)vote));
        else atomicMin(&s_pick_min, wbase + __ffs((int)vote) - 1);
    }
    __syncthreads();
    int pick = fb ? s_pick_max : s_pick_min;
    if (pick < 0 || pick >= kVT) pick = kVT - 1;
    // ---- and the element: the picked thread's words go to shared memory
    // and the first warp walks them, EPT / 32 elements (at least one) a lane
    if ((int)threadIdx.x == pick) {
#pragma unroll
        for (int k = 0; k < kResLoadsPerThread; ++k) {
            s_words[0][k] = rt[k];
            s_words[1][k] = rd[k];
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        constexpr int EPL = EPT >= 32 ? EPT / 32 : 1;
        const int lane = threadIdx.x;
        const int f0p = cstar * p.res_chunk_elems + pick * EPT;
        const int fnp = max(0, min(EPT, a.V - f0p));
        float wv[EPL], lsum = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int j = lane * EPL + e;
            wv[e] = j < fnp ? elem_weight<T>(rw, mode, smem_elem<T>(s_words[0], j),
                                             mode == 0 ? smem_elem<T>(s_words[1], j) : 0.f)
                            : 0.f;
            lsum = __fadd_rn(lsum, wv[e]);
        }
        // the weight before this lane's elements (lanes in order), after the
        // prefix of the threads before the picked one
        float incl_l = lsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl_l, off);
            if (lane >= off) incl_l = __fadd_rn(incl_l, t);
        }
        float acc = __fadd_rn(base, pick > 0 ? s_prefix[pick - 1] : 0.f);
        acc = __fadd_rn(acc, __fsub_rn(incl_l, lsum));
        int hit_e = -1, last_e = -1;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            acc = __fadd_rn(acc, wv[e]);
            if (hit_e < 0 && lane * EPL + e < fnp && acc > theta) hit_e = e;
            if (wv[e] > 0.f) last_e = e;
        }
        const unsigned hv = __ballot_sync(0xffffffffu, hit_e >= 0);
        const unsigned pv = __ballot_sync(0xffffffffu, last_e >= 0);
        int y;
        if (!fb && hv != 0u) {
            const int l = __ffs((int)hv) - 1;  // the first crossing
            y = f0p + l * EPL + __shfl_sync(0xffffffffu, hit_e, l);
        } else if (pv != 0u) {
            const int l = 31 - __clz((int)pv);  // no crossing: the last element with weight
            y = f0p + l * EPL + __shfl_sync(0xffffffffu, last_e, l);
        } else {
            y = max(f0p, 0);
        }
        if (lane == 0) {
            a.out_tokens[(size_t)b * (a.N + 1) + d.a] = y;
            if (!CLUSTER) w.counters[a.B + b] = 0;  // ready for the next call
        }
    }
}

// ---------------------------------------------------------------- tree greedy

// Shared state of the greedy walk over one sequence's tree.
struct TreeWalkSmem {
    int am[kMaxTreeT], par[kMaxTreeT], tok[kMaxTreeT], depth[kMaxTreeT], path[kMaxTreeT];
    unsigned char ok[kMaxTreeT];
    int best, bad, tb_raw;
    int prefix_len;  // fused step: L_b, read with the other inputs
    int red[kVWarps];
};

// The walk's inputs of sequence b -- parents, node tokens, node count -- into
// shared memory, by the whole CTA (a barrier must follow before they are read).
__device__ __forceinline__ void tree_walk_load(const TreeArgs &a, int b, TreeWalkSmem &ts) {
    for (int i = threadIdx.x; i < a.T; i += kVT) {
        ts.par[i] = a.parents ? a.parents[(size_t)b * a.T + i] : i - 1;  // NULL: a chain
        ts.tok[i] = a.tokens[(size_t)b * a.T + i];
    }
    if (threadIdx.x == 0) ts.tb_raw = a.node_counts ? a.node_counts[b] : a.T;
    if (threadIdx.x == 32 && a.hook.step_ctr) ts.prefix_len = a.hook.prefix_lens[b];
}

// Greedy longest agreeing path of sequence b from the target's argmax per
// node (ts.am, -1 for none) and the inputs tree_walk_load brought in, by a
// whole CTA of kVT threads: validation, the walk in node order, then the
// outputs.  `late`: the statistics pass gave up, so no decision is taken.
__device__ __forceinline__ void tree_walk(const TreeArgs &a, int b, bool late, TreeWalkSmem &ts) {
    __syncthreads();
    const int tid = threadIdx.x;
    // this sequence's nodes; those past T_b are padding
    const int tb_raw = ts.tb_raw;
    const bool tb_bad = late || ts.par[0] != -1 || tb_raw < 1 || tb_raw > a.T;
    const int Tb = tb_bad ? 1 : tb_raw;
    int bad = tb_bad;
    for (int i = tid; i < Tb; i += kVT)
        if (i > 0 && (ts.par[i] < 0 || ts.par[i] >= i || ts.tok[i] < 0 || ts.tok[i] >= a.V)) bad = 1;
    bad = __syncthreads_or(bad);
    // Every node at once: a thread follows its nodes' parent chains (parents
    // precede their children, so a chain ends at the root after depth steps):
    // ok = every node on the chain holds the target's argmax at its parent.
    // The deepest ok node wins, the smallest index among equal depths: the
    // largest key depth * 1024 + (1023 - node).
    int key = -1;
    if (!bad) {
        for (int i = tid; i < Tb; i += kVT) {
            int node = i, d = 0;
            bool okc = true;
            while (node > 0) {
                const int pa = ts.par[node];
                okc = okc && ts.tok[node] == ts.am[pa];
                node = pa;
                ++d;
            }
            ts.depth[i] = d;
            ts.ok[i] = okc;
            if (okc) key = max(key, d * 1024 + (1023 - i));
        }
    }
    key = __reduce_max_sync(0xffffffffu, key);
    if ((tid & 31) == 0) ts.red[tid >> 5] = key;
    __syncthreads();
    if (tid == 0) {
        int k = ts.red[0];
        for (int w = 1; w < kVWarps; ++w) k = max(k, ts.red[w]);
        int bst = 0;
        if (!bad) {
            bst = 1023 - (k & 1023);  // the root is always ok: k >= 1023
            int node = bst;
            for (int dd = k >> 10; dd >= 0; --dd) {
                ts.path[dd] = node;
                node = ts.par[node];
            }
        }
        ts.bad = bad;
        ts.best = bst;
        a.accepted_len[b] = bad ? -1 : ts.depth[bst];
        if (a.seq_status) a.seq_status[b] = late ? SV_ERR_TIMEOUT : bad ? SV_ERR_BAD_INPUT : SV_OK;
    }
    __syncthreads();
    const int depth = ts.bad ? -1 : ts.depth[ts.best];
    for (int i = threadIdx.x; i < a.T; i += kVT) {
        int pn = -1, ot = -1;
        if (i <= depth) {
            pn = ts.path[i];
            ot = i < depth ? ts.tok[ts.path[i + 1]] : ts.am[ts.best];
        }
        a.path_nodes[(size_t)b * a.T + i] = pn;
        a.out_tokens[(size_t)b * a.T + i] = ot;
    }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kVT) tree_stats_kernel(TreeArgs a, VocabPlan p, WsView w) {
    __shared__ float4 scratch[kVWarps];
    __shared__ int s_last;
    __shared__ TreeWalkSmem ts;

    const int per_seq = a.T * p.nchunks;
    const int item = blockIdx.x;
    const int b = item / per_seq;
    const int rem = item - b * per_seq;
    const int r = rem / p.nchunks;
    const int c = rem - r * p.nchunks;
    const T *row = static_cast<const T *>(a.target) + ((size_t)b * a.T + r) * a.V;
    const int begin = c * p.chunk_elems;
    const int end = min(a.V, begin + p.chunk_elems);

    griddep_wait();
    griddep_launch_dependents();
    float best = kNegInf;
    int idx = INT_MAX;
    // a padding node's row (past T_b) is never read
    const bool pad_row = a.node_counts != nullptr && r > 0 && r >= a.node_counts[b];
    if (!pad_row) chunk_thread_argmax<T, VEC>(row, begin, end, best, idx);
    float m = 0.f, s = 0.f;
    cta_reduce_stats<true>(m, s, best, idx, scratch);
    if (threadIdx.x == 0) {
        RowPartial out;
        out.m = 0.f;
        out.s = 0.f;
        out.best = best;
        out.idx = idx;
        w.partials[item] = out;
        __threadfence();
        const int old = atomicAdd(&w.counters[b], 1);
        s_last = (old == per_seq - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of sequence b: argmax per node, then the greedy walk
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int rr = warp; rr < a.T; rr += kVWarps) {
        const RowPartial rp = warp_merge_row<true>(
            w.partials + (size_t)b * per_seq + (size_t)rr * p.nchunks, p.nchunks);
        if (lane == 0) ts.am[rr] = rp.idx == INT_MAX ? -1 : rp.idx;
    }
    tree_walk_load(a, b, ts);
    tree_walk(a, b, false, ts);
    if (threadIdx.x == 0) w.counters[b] = 0;  // ready for the next call
}

// ---------------------------------------------------------------- tree greedy, streaming form

// Rows 16-byte aligned: the argmax pass as a persistent grid streaming the
// units (sequence, node row, 32 KB chunk) of a balanced contiguous range
// through the same ring of bulk copies as the chain statistics (evict-first).
// Each consumer warp reduces an eighth of a unit to (largest value, smallest
// index holding it) -- the packed maximum first, then the first element
// equal to it -- and leaves one record.  The walk is the next kernel's.
// Rows of padding nodes (past T_b) are not read.
// Units a producer claims at a time from the pass's shared counter.
constexpr int kSClaim = 4;

template <typename T>
__global__ void __launch_bounds__(kSThreads, 1)
    tree_stats_stream_kernel(TreeArgs a, VocabPlan p, WsView w) {
    SV_SPAN(kSpanTreeStats);
    extern __shared__ __align__(128) uint8_t ring[];  // kSStages * kSUnitBytes
    __shared__ uint64_t full[kSStages], empty[kSStages];
    __shared__ int unit_of[kSStages];  // the unit in each stage; -1: no more units
    constexpr int PV = Elem<T>::kPerVec;
    constexpr int kUnitElems = kSUnitBytes / (int)sizeof(T);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_seq = a.T * p.nchunks;
    const int U = a.B * per_seq;  // units (the launch keeps this below 2^31)
    float2 *rec = reinterpret_cast<float2 *>(w.partials);  // [B][T][nchunks][kSGroupWarps]
    int *timed_out = w.counters + 2 * a.B;
    // The CTAs claim units kSClaim at a time from one counter (the walk
    // clears it), so that CTAs that start late -- behind an attention kernel
    // whose CTAs end at different times -- take fewer of them.
    int *claim = w.counters + 2 * a.B + 1;
    // node r of sequence b is read unless it is padding (node 0 always is read)
    auto row_in_use = [&](int b, int r) {
        return r == 0 || a.node_counts == nullptr || r < a.node_counts[b];
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSGroupWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    if (warp == kSWarps) {
        // ================= producer: one bulk copy per unit
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            long long k = 0;
            int next = 0, lim = 0;  // the claimed units not yet issued
            int ends = 0;           // "no more units" stages published: one per consumer group
            while (ends < 2) {
                const int s = (int)(k % kSStages);
                if (!mbar_wait_bounded(&empty[s], (uint32_t)(((k / kSStages) & 1) ^ 1))) {
                    atomicExch(timed_out, 1);  // a stage never came free
                    break;
                }
                if (next == lim && ends == 0) {
                    next = atomicAdd(claim, kSClaim);
                    lim = min(next + kSClaim, U);
                }
                if (next >= lim) {  // the units are all claimed: an end marker, no copy
                    unit_of[s] = -1;
                    ++ends;
                    mbar_arrive(&full[s]);
                    ++k;
                    continue;
                }
                const int u = next++;
                unit_of[s] = u;
                const int b = u / per_seq;
                const int rem = u - b * per_seq;
                const int r = rem / p.nchunks, c = rem - r * p.nchunks;
                if (!row_in_use(b, r)) {  // padding: the stage's phase, no copy
                    mbar_arrive(&full[s]);
                    ++k;
                    continue;
                }
                const T *row = static_cast<const T *>(a.target) + ((size_t)b * a.T + r) * a.V;
                const int begin = c * kUnitElems;
                const uint32_t bytes = (uint32_t)(min(kUnitElems, a.V - begin) * (int)sizeof(T));
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_load_hint(ring + s * kSUnitBytes, row + begin, bytes, &full[s], pol);
                ++k;
            }
            // every copy issued must land before the CTA may exit
            const long long first = k > kSStages ? k - kSStages : 0;
            for (long long j = first; j < k; ++j)
                mbar_wait_bounded(&full[j % kSStages], (uint32_t)((j / kSStages) & 1));
        }
        return;
    }

    // ================= consumers: two groups of eight warps, alternate stages
    const int grp = (warp >> 2) & 1, gw = ((warp >> 3) << 2) | (warp & 3);
    for (long long k = grp;; k += 2) {
        const int s = (int)(k % kSStages);
        if (!warp_wait_bounded(&full[s], (uint32_t)((k / kSStages) & 1))) {
            if (lane == 0) atomicExch(timed_out, 1);  // records left unwritten
            break;
        }
        const int u = unit_of[s];
        if (u < 0) break;  // no more units
        const int b = u / per_seq;
        const int rem = u - b * per_seq;
        const int r = rem / p.nchunks, c = rem - r * p.nchunks;
        const int n = min(kUnitElems, a.V - c * kUnitElems);  // elements in this unit (a multiple of PV)
        float2 *dst = rec + (((size_t)b * a.T + r) * p.nchunks + c) * kSGroupWarps + gw;
        if (!row_in_use(b, r)) {  // padding: nothing landed, an empty record
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                *dst = make_float2(kNegInf, __int_as_float(INT_MAX));
            }
            continue;
        }
        uint4 buf[kSWordsPerLane];
#pragma unroll
        for (int q = 0; q < kSWordsPerLane; ++q) {
            const int wi = (gw * kSWordsPerLane + q) * 32 + lane;  // 16-byte word of the unit
            buf[q] = wi * PV < n ? *reinterpret_cast<const uint4 *>(ring + s * kSUnitBytes + wi * 16)
                                 : neg_inf_vec<T>();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the words are in registers
        // the lane's largest value and the first of its words holding it
        // (words in index order; NaN never wins), then the warp's maximum and
        // the smallest index holding it: only the winning word is unpacked
        float best = kNegInf;
        int bq = 0;
#pragma unroll
        for (int q = 0; q < kSWordsPerLane; ++q) {
            const float mq = word_max<T>(buf[q]);
            if (mq > best) {
                best = mq;
                bq = q;
            }
        }
        float vmax = best;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        int idx = INT_MAX;
        if (vmax != kNegInf && best == vmax) {  // this lane holds the maximum
            uint4 wq = buf[0];
#pragma unroll
            for (int q = 1; q < kSWordsPerLane; ++q)
                if (q == bq) wq = buf[q];
            float x[PV];
            Elem<T>::unpack(wq, x);
            const int e0 = c * kUnitElems + ((gw * kSWordsPerLane + bq) * 32 + lane) * PV;
#pragma unroll
            for (int j = PV - 1; j >= 0; --j)
                if (x[j] == vmax) idx = e0 + j;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, off));
        if (lane == 0) *dst = make_float2(vmax, __int_as_float(idx));
    }
}

// Fused tree step: the walk's half of the compaction.  It writes the new
// cache length, then arrives on the counter of every KV head of sequence b;
// for each head where it arrives last (the attention has read that head's
// rows) it moves the path's rows itself: rows L + path[d] -> L + d, d = 1..a,
// K and V, every source read into registers before any row is written.
constexpr int kMaxStepHkv = 256;
constexpr int kStepRowWords = 16;  // 16-byte words of a 128-dim bf16 row
constexpr int kStepMoveRegs = 8;   // words a thread holds: 256 * 8 >= 63 rows * 2 * 16
static_assert(kVT * kStepMoveRegs >= (kStepHookMaxT - 1) * 2 * kStepRowWords,
              "the walk cannot hold the accepted rows the hook allows");

__device__ __forceinline__ void step_hook_arrive(const TreeArgs &a, int b, const TreeWalkSmem &ts) {
    __shared__ unsigned char s_last[kMaxStepHkv];
    __shared__ int s_any;
    const StepHook &h = a.hook;
    const int acc = ts.bad ? -1 : ts.depth[ts.best];
    const int L = ts.prefix_len;
    const int tb_raw = ts.tb_raw;
    const bool fits = L >= 0 && tb_raw >= 1 && tb_raw <= a.T && (long long)L + tb_raw <= h.S_max;
    if (threadIdx.x == 0) {
        h.new_kv_lens[b] = (fits && acc >= 0) ? L + acc + 1 : L;
        s_any = 0;
    }
    __threadfence();  // this thread's path and token writes, before the arrivals
    __syncthreads();
    for (int hh = threadIdx.x; hh < h.Hkv; hh += kVT) {
        const int old = atomicAdd(h.step_ctr + (size_t)b * h.Hkv + hh, 1);
        s_last[hh] = old == h.rg_count;
        if (old == h.rg_count) s_any = 1;
    }
    __syncthreads();
    if (!s_any) return;
    __threadfence();  // the attention has finished with these rows
    const bool move = fits && acc > 0;
    for (int hh = 0; hh < h.Hkv; ++hh) {
        if (!s_last[hh]) continue;
        if (move) {
            const size_t head = ((size_t)b * h.Hkv + hh) * h.S_max;
            const int n = acc * 2 * kStepRowWords;
            uint4 reg[kStepMoveRegs];
#pragma unroll
            for (int k = 0; k < kStepMoveRegs; ++k) {
                const int wi = threadIdx.x + k * kVT;
                if (wi < n) {
                    const int d = 1 + wi / (2 * kStepRowWords), kv = (wi / kStepRowWords) & 1;
                    reg[k] = (kv ? h.v : h.k)[(head + L + ts.path[d]) * kStepRowWords + wi % kStepRowWords];
                }
            }
            __syncthreads();  // every source of this head is read
#pragma unroll
            for (int k = 0; k < kStepMoveRegs; ++k) {
                const int wi = threadIdx.x + k * kVT;
                if (wi < n) {
                    const int d = 1 + wi / (2 * kStepRowWords), kv = (wi / kStepRowWords) & 1;
                    if (ts.path[d] != d)
                        (kv ? h.v : h.k)[(head + L + d) * kStepRowWords + wi % kStepRowWords] = reg[k];
                }
            }
        }
        if (threadIdx.x == 0) h.step_ctr[(size_t)b * h.Hkv + hh] = 0;  // ready for the next call
    }
}

// The greedy walk after the streaming argmax pass: one CTA per sequence
// merges each node row's records into the row's argmax, then walks.
template <typename T>
__global__ void __launch_bounds__(kVT) tree_decide_kernel(TreeArgs a, VocabPlan p, WsView w) {
    SV_SPAN(kSpanTreeDecide);
    __shared__ TreeWalkSmem ts;
    const int b = blockIdx.x;
    // The tree and its tokens are inputs of the call, not outputs of the
    // argmax pass: they are read while that pass still runs (this grid starts
    // only after the pass has passed its own wait for the work before the
    // call, so they are complete); only the records wait for the pass.
    tree_walk_load(a, b, ts);
    griddep_wait();
    griddep_launch_dependents();
    if (b == 0 && threadIdx.x == 0) w.counters[2 * a.B + 1] = 0;  // the pass's claim counter, for the next call
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_row = p.nchunks * kSGroupWarps;
    const float2 *rec = reinterpret_cast<const float2 *>(w.partials) + (size_t)b * a.T * per_row;
    // a warp per row, four rows of a warp with their loads in flight together
    for (int r0 = warp; r0 < a.T; r0 += 4 * kVWarps) {
        float best[4];
        int idx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            best[q] = kNegInf;
            idx[q] = INT_MAX;
        }
        for (int i0 = 0; i0 < per_row; i0 += 32) {
            float2 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = r0 + q * kVWarps, i = i0 + lane;
                v[q] = (rr < a.T && i < per_row) ? __ldcg(rec + (size_t)rr * per_row + i)
                                                 : make_float2(kNegInf, __int_as_float(INT_MAX));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) merge_argmax(best[q], idx[q], v[q].x, __float_as_int(v[q].y));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float b2 = __shfl_xor_sync(0xffffffffu, best[q], off);
                const int i2 = __shfl_xor_sync(0xffffffffu, idx[q], off);
                merge_argmax(best[q], idx[q], b2, i2);
            }
            const int rr = r0 + q * kVWarps;
            if (lane == 0 && rr < a.T) ts.am[rr] = idx[q] == INT_MAX ? -1 : idx[q];
        }
    }
    const bool late = __ldcg(w.counters + 2 * a.B) != 0;
    tree_walk(a, b, late, ts);
    if (a.hook.step_ctr) step_hook_arrive(a, b, ts);
}

// ---------------------------------------------------------------- stochastic tree

// Multi-draft speculative sampling on a tree (the SpecInfer rule: the pages,
// "Chapitre 9 -- Décodage spéculatif" §9.2, have the target choose among
// drafted paths without giving a rule).  Node u's children were drawn from
// q_u = softmax(draft row u); the target's distribution is p_u.  From the
// root, the children of u are tried in index order against the residual
// max(0, p_u - c q_u) / N(c), N(c) = sum_v max(0, p_u(v) - c q_u(v)), c = 0 at
// the first child: child v (token x) is accepted iff
// u_accept[v] * q_u(x) * N(c) < max(0, p_u(x) - c q_u(x)); a rejection sets
// c = c + N(c) (the rejection step applied to the residual, in closed form).
// With no child accepted, or at a leaf, the final token is drawn from
// max(0, p_u - c q_u) (p_u when that sums to zero).
//
// Kernel 1: the (max, sum) records of every target row and of the draft row of
// every node with children, one CTA per (row, chunk).  Kernel 2: one
// thread-block cluster per sequence walks the tree.  Every CTA of the cluster
// takes the same decisions from the same inputs; each N(c) and the final draw
// are passes over the row pair in which every thread sums its own contiguous
// segment of the vocabulary (CTA rank, then thread, then element: index
// order), the CTAs' partial sums meeting in distributed shared memory.

constexpr int kWT = 256;                  // threads of a walking CTA
constexpr int kWWarps = kWT / 32;
constexpr int kWClusterMax = 16;          // CTAs of a walking cluster (16: non-portable)
constexpr int kMaxWSeg = 4096;            // elements a thread owns in a pass

template <typename T, bool VEC>
__global__ void __launch_bounds__(kVT) stree_stats_kernel(STreeArgs a, VocabPlan p, float2 *rec) {
    __shared__ float red[2 * kVWarps];
    const int per_seq = 2 * a.T * p.nchunks;
    const int item = blockIdx.x;
    const int b = item / per_seq;
    const int rem = item - b * per_seq;
    const int r = rem / p.nchunks;  // rows 0..T-1 target, T..2T-1 draft
    const int c = rem - r * p.nchunks;
    griddep_wait();
    griddep_launch_dependents();
    // this sequence's nodes (an invalid count is reported by the walk)
    const int tb_raw = a.node_counts ? a.node_counts[b] : a.T;
    const int tb = (tb_raw >= 1 && tb_raw <= a.T) ? tb_raw : a.T;
    const int u = r < a.T ? r : r - a.T;
    bool used = u < tb;
    if (used && r >= a.T) {  // a draft row is read only for a node with children
        int has_child = 0;
        for (int v = u + 1 + (int)threadIdx.x; v < tb; v += kVT)
            if ((a.parents ? a.parents[(size_t)b * a.T + v] : v - 1) == u) has_child = 1;
        used = __syncthreads_or(has_child) != 0;
    }
    if (!used) {  // a padding node's row, a leaf's draft row: not read
        if (threadIdx.x == 0) rec[item] = make_float2(kNegInf, 0.f);
        return;
    }
    const T *row = r < a.T ? static_cast<const T *>(a.target) + ((size_t)b * a.T + r) * a.V
                           : static_cast<const T *>(a.draft) + ((size_t)b * a.T + (r - a.T)) * a.V;
    const int begin = c * p.chunk_elems;
    const int end = min(a.V, begin + p.chunk_elems);
    float m = 0.f, s = 0.f;
    chunk_cta_stats<T, VEC>(row, begin, end, red, m, s);
    if (threadIdx.x == 0) rec[item] = make_float2(m, s);
}

// Sum over the CTA of one value per thread, in a fixed order (warp shuffles,
// then the warps in order); every thread gets the total.
__device__ __forceinline__ float walk_block_sum(float v, float *red /* [kWWarps] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWWarps; ++w) t += red[w];
    return t;
}

// p_u and q_u of one element (the same arithmetic everywhere in the walk).
struct STreeRow {
    float mt, it, md, id;  // log2-domain maxima and reciprocal sums of the target and draft rows
    __device__ __forceinline__ float p(float lt) const {
        return __fmul_rn(ex2_approx(__fmaf_rn(lt, kLog2e, -mt)), it);
    }
    __device__ __forceinline__ float q(float ld) const {
        return __fmul_rn(ex2_approx(__fmaf_rn(ld, kLog2e, -md)), id);
    }
};

// Elements [e0, e1) of the thread's segment in index order: their weights
// summed one by one (words of 8 or 4 elements when the rows are 16-byte
// aligned), or, with `want` in range, the first element where `acc` plus the
// running sum passes `theta` (and the last element with weight) -- the same
// additions in the same order either way.
template <typename T, bool VEC>
__device__ __forceinline__ float stree_seg(const T *trow, const T *drow, const STreeRow &rs, float c,
                                           int e0, int e1, float acc, float theta, int *hit,
                                           int *last) {
    constexpr int PV = Elem<T>::kPerVec;
    float s = acc;
    for (int e = e0; e < e1; e += PV) {
        float xt[PV], xd[PV];
        if (VEC && e + PV <= e1) {
            Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(trow + e)), xt);
            if (c != 0.f) Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(drow + e)), xd);
        } else {
#pragma unroll
            for (int j = 0; j < PV; ++j) {
                xt[j] = e + j < e1 ? Elem<T>::at(trow, e + j) : kNegInf;
                xd[j] = (c != 0.f && e + j < e1) ? Elem<T>::at(drow, e + j) : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < PV; ++j) {
            if (e + j >= e1) break;
            const float pe = rs.p(xt[j]);
            const float w = c == 0.f ? pe : fmaxf(__fsub_rn(pe, __fmul_rn(c, rs.q(xd[j]))), 0.f);
            s = __fadd_rn(s, w);
            if (hit) {
                if (w > 0.f) *last = e + j;
                if (*hit < 0 && s > theta) *hit = e + j;
            }
        }
    }
    return s;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kWT) stree_walk_kernel(STreeArgs a, VocabPlan p, const float2 *rec) {
    __shared__ int s_par[kMaxTreeT], s_tok[kMaxTreeT], s_kids[kMaxTreeT];
    __shared__ unsigned char s_child[kMaxTreeT];
    __shared__ float2 s_ms[2][kMaxTreeT];  // merged (max, sum) of the target / draft row of each node
    __shared__ float s_red[kWWarps];
    __shared__ float s_part[2];            // this CTA's partial sum of a pass (two in turn)
    __shared__ int s_bad, s_nkids, s_next, s_pick;
    __shared__ float s_prefix[kWT];
    // for each node v: its acceptance uniform, and the target and draft logits
    // of its token at its parent (gathered once, so a child's test reads no memory)
    __shared__ float s_ua[kMaxTreeT], s_lt[kMaxTreeT], s_ld[kMaxTreeT];
    griddep_wait();
    griddep_launch_dependents();
    const int C = p.walk_cluster;
    const int rank = (int)cluster_ctarank();
    const int b = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nT = a.T, V = a.V;
    // this sequence's nodes; those past T_b are padding
    const int tb_raw = a.node_counts ? a.node_counts[b] : nT;
    const bool tb_ok = tb_raw >= 1 && tb_raw <= nT;
    const int nb = tb_ok ? tb_raw : 1;
    for (int i = tid; i < nb; i += kWT) {
        s_par[i] = a.parents ? a.parents[(size_t)b * nT + i] : i - 1;  // NULL: a chain
        s_tok[i] = a.tokens[(size_t)b * nT + i];
        s_ua[i] = i > 0 ? a.u_accept[(size_t)b * nT + i] : 0.f;
        s_child[i] = 0;
    }
    if (tid == 0) s_bad = tb_ok ? 0 : 1;
    // merge the records of the target and draft rows of the first T_b nodes
    // (a row that is not read has the empty record): a thread a row, its
    // chunks in order, eight records in flight (short code: it runs once per
    // launch, fetched cold)
    for (int rr = tid; rr < 2 * nT; rr += kWT) {
        const int u = rr < nT ? rr : rr - nT;
        if (u >= nb) continue;
        const float2 *r0 = rec + ((size_t)b * 2 * nT + rr) * p.nchunks;
        float m = kNegInf, s = 0.f;
        for (int c0 = 0; c0 < p.nchunks; c0 += 8) {
            float2 r2[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                r2[j] = c0 + j < p.nchunks ? __ldcg(r0 + c0 + j) : make_float2(kNegInf, 0.f);
#pragma unroll
            for (int j = 0; j < 8; ++j) merge_ms(m, s, r2[j].x, r2[j].y);
        }
        s_ms[rr < nT ? 0 : 1][u] = make_float2(m, s);
    }
    __syncthreads();
    for (int i = 1 + tid; i < nb; i += kWT) {
        const int pa = s_par[i], x = s_tok[i];
        if (pa < 0 || pa >= i || x < 0 || x >= V) {
            s_bad = 1;
        } else {
            s_child[pa] = 1;
            s_lt[i] = Elem<T>::at(static_cast<const T *>(a.target) + ((size_t)b * nT + pa) * V, x);
            s_ld[i] = Elem<T>::at(static_cast<const T *>(a.draft) + ((size_t)b * nT + pa) * V, x);
        }
    }
    if (tid == 0 && s_par[0] != -1) s_bad = 1;
    __syncthreads();
    // a used row (every target row, the draft rows of nodes with children)
    // without a finite distribution is bad input
    auto finite_ms = [](float2 v) { return isfinite(v.x) && isfinite(v.y) && v.y > 0.f; };
    for (int u = tid; u < nb; u += kWT)
        if (!finite_ms(s_ms[0][u]) || (s_child[u] && !finite_ms(s_ms[1][u]))) s_bad = 1;
    __syncthreads();
    // every CTA reaches the same verdict from the same inputs, so all of them
    // take the same path through the cluster barriers below
    const bool bad = s_bad != 0;
    // this thread's segment of the vocabulary (a multiple of 8 elements long):
    // CTA rank, then thread, in index order
    const int seg = ((V + C * kWT - 1) / (C * kWT) + 7) & ~7;
    const int gt = rank * kWT + tid;
    const int e0 = min(V, gt * seg), e1 = min(V, e0 + seg);
    int pass = 0;
    // the cluster's sum of one value per thread: CTA sums in a fixed order,
    // then the CTAs in rank order (every CTA gets the same total)
    // (lane k of every warp reads CTA k's sum, all C loads in flight together;
    // `part` keeps it for the final draw's search)
    float part = 0.f;
    auto cluster_total = [&](float v, float *cta_total) -> float {
        const float t = walk_block_sum(v, s_red);
        if (cta_total) *cta_total = t;
        if (tid == 0) s_part[pass & 1] = t;
        cluster_sync();
        part = lane < C ? ld_shared_cluster_f32(&s_part[pass & 1], (uint32_t)lane) : 0.f;
        float tot = 0.f;
        for (int k = 0; k < C; ++k) tot = __fadd_rn(tot, __shfl_sync(0xffffffffu, part, k));
        ++pass;  // the other buffer next: a CTA may run ahead into the next pass
        return tot;
    };
    int depth = 0, u = 0;
    if (!bad) {
        for (int step = 0; step < nb; ++step) {
            // children of u in index order (warp 0, 32 nodes a ballot)
            if (warp == 0) {
                int n = 0;
                for (int v0 = u + 1; v0 < nb; v0 += 32) {
                    const bool kid = v0 + lane < nb && s_par[v0 + lane] == u;
                    const unsigned mk = __ballot_sync(0xffffffffu, kid);
                    if (kid) s_kids[n + __popc(mk & ((1u << lane) - 1u))] = v0 + lane;
                    n += __popc(mk);
                }
                if (lane == 0) {
                    s_nkids = n;
                    s_next = -1;
                }
            }
            __syncthreads();
            const int nk = s_nkids;
            const T *trow = static_cast<const T *>(a.target) + ((size_t)b * nT + u) * V;
            const T *drow = static_cast<const T *>(a.draft) + ((size_t)b * nT + u) * V;
            STreeRow rs;
            rs.mt = s_ms[0][u].x;
            rs.it = __frcp_rn(s_ms[0][u].y);
            rs.md = nk > 0 ? s_ms[1][u].x : 0.f;
            rs.id = nk > 0 ? __frcp_rn(s_ms[1][u].y) : 0.f;
            float c = 0.f;
            for (int i = 0; i < nk; ++i) {
                // N(c): 1 for c = 0, else a pass over the row pair
                const float n = c == 0.f ? 1.f
                                         : cluster_total(stree_seg<T, VEC>(trow, drow, rs, c, e0, e1, 0.f,
                                                                           0.f, nullptr, nullptr),
                                                         nullptr);
                const int v = s_kids[i];
                if (tid == 0) {
                    const float px = __fdiv_rn(exp2_diff_accurate(s_lt[v], rs.mt), s_ms[0][u].y);
                    const float qx = __fdiv_rn(exp2_diff_accurate(s_ld[v], rs.md), s_ms[1][u].y);
                    const float r = fmaxf(__fsub_rn(px, __fmul_rn(c, qx)), 0.f);
                    const float lhs = __fmul_rn(__fmul_rn(s_ua[v], qx), n);
                    if (lhs < r) s_next = v;
                }
                __syncthreads();
                if (s_next >= 0) break;
                c = __fadd_rn(c, n);
            }
            const int next = s_next;
            if (next >= 0) {
                u = next;
                ++depth;
                if (tid == 0 && rank == 0) {
                    a.path_nodes[(size_t)b * nT + depth] = u;
                    a.out_tokens[(size_t)b * nT + depth - 1] = s_tok[u];
                }
                __syncthreads();  // s_next and s_kids are rewritten for the next node
                continue;
            }
            // ---- the final draw: the CTA totals, the CTA, the thread, the element
            float ts = stree_seg<T, VEC>(trow, drow, rs, c, e0, e1, 0.f, 0.f, nullptr, nullptr);
            float cta = 0.f;
            float S = cluster_total(ts, &cta);
            if (!(S > 0.f)) {  // the residual vanished: draw from p_u
                c = 0.f;
                ts = stree_seg<T, VEC>(trow, drow, rs, c, e0, e1, 0.f, 0.f, nullptr, nullptr);
                S = cluster_total(ts, &cta);
            }
            const float theta = __fmul_rn(a.u_sample[b], S);
            // the CTA where the cluster prefix passes theta (rank order; the
            // same search in every CTA)
            int kstar = -1, klast = 0;
            float base = 0.f, run = 0.f;
            for (int k = 0; k < C; ++k) {
                const float t = __shfl_sync(0xffffffffu, part, k);  // CTA k's sum in the last pass
                if (t > 0.f) klast = k;
                const float nb2 = __fadd_rn(run, t);
                if (kstar < 0 && nb2 > theta) {
                    kstar = k;
                    base = run;
                }
                run = nb2;
            }
            bool fallback = false;
            if (kstar < 0) {  // rounding left no crossing: the last CTA with weight
                fallback = true;
                kstar = klast;
                base = 0.f;
                for (int k = 0; k < kstar; ++k) base = __fadd_rn(base, __shfl_sync(0xffffffffu, part, k));
            }
            if (rank == kstar) {
                // inclusive prefix of this CTA's thread sums (warp scan, then the warps in order)
                float incl = ts;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl = __fadd_rn(incl, t);
                }
                __syncthreads();  // the last block sum's readers are done with s_red
                if (lane == 31) s_red[warp] = incl;
                if (tid == 0) s_pick = kWT;
                __syncthreads();
                float wbase = 0.f;
                for (int w = 0; w < warp; ++w) wbase = __fadd_rn(wbase, s_red[w]);
                incl = __fadd_rn(wbase, incl);
                s_prefix[tid] = incl;
                if (!fallback && __fadd_rn(base, incl) > theta) atomicMin(&s_pick, tid);
                __syncthreads();
                int pick = s_pick;
                if (pick >= kWT) {  // no crossing: the last thread holding weight
                    pick = 0;
                    for (int t2 = kWT - 1; t2 > 0; --t2)
                        if (s_prefix[t2] > s_prefix[t2 - 1]) {
                            pick = t2;
                            break;
                        }
                }
                if (tid == pick) {
                    const int gp = rank * kWT + pick;
                    const int p0 = min(V, gp * seg), p1 = min(V, p0 + seg);
                    int y = -1, last = -1;
                    stree_seg<T, VEC>(trow, drow, rs, c, p0, p1,
                                      __fadd_rn(base, pick > 0 ? s_prefix[pick - 1] : 0.f),
                                      fallback ? __int_as_float(0x7f800000) : theta, &y, &last);
                    if (y < 0) y = last >= 0 ? last : max(p0, 0);
                    a.out_tokens[(size_t)b * nT + depth] = y;
                }
            }
            break;
        }
    }
    cluster_sync();  // no CTA leaves while another may still read its partial sums
    if (rank != 0) return;
    __syncthreads();
    // outputs: the path and tokens past the end, the length and the status
    for (int i = tid; i < nT; i += kWT) {
        if (bad || i > depth) a.path_nodes[(size_t)b * nT + i] = -1;
        if (bad || i > depth) a.out_tokens[(size_t)b * nT + i] = -1;
    }
    if (tid == 0) {
        if (!bad) a.path_nodes[(size_t)b * nT] = 0;
        a.accepted_len[b] = bad ? -1 : depth;
        if (a.seq_status) a.seq_status[b] = bad ? SV_ERR_BAD_INPUT : SV_OK;
    }
}

// ---------------------------------------------------------------- host side

VocabPlan plan_vocab(bool chain, int B, int rows_or_n, int V, int dtype) {
    VocabPlan p{};
    const int esz = dtype == SV_F32 ? 4 : 2;
    const int per_vec = 16 / esz;
    p.rows_per_seq = chain ? 2 * rows_or_n + 1 : rows_or_n;
    p.chunk_elems = kVT * kLoadsPerThread * per_vec;
    p.nchunks = (V + p.chunk_elems - 1) / p.chunk_elems;
    p.res_chunk_elems = kVT * kResLoadsPerThread * per_vec;
    p.res_chunks = chain ? (V + p.res_chunk_elems - 1) / p.res_chunk_elems : 0;
    p.vec = ((size_t)V * esz) % 16 == 0;
    p.recs_per_unit = p.vec ? kSGroupWarps : 1;
    size_t off = 0;
    p.off_counters = off;
    off = align_up(off + sizeof(int) * (2 * (size_t)B + 4), 256);
    p.off_partials = off;  // tree: a RowPartial per (row, chunk); chain: recs_per_unit (max, sum) records
    const size_t per_unit = chain ? sizeof(float2) * p.recs_per_unit
                                  : (p.vec ? sizeof(float2) * kSGroupWarps : sizeof(RowPartial));
    off = align_up(off + per_unit * (size_t)B * p.rows_per_seq * p.nchunks, 256);
    p.off_chunktot = off;
    off = align_up(off + (chain ? sizeof(float2) * (size_t)B * p.res_chunks : 0), 256);
    p.bytes = off;
    return p;
}

// How many clusters of `size` CTAs of `threads` threads of `fn` this device
// holds at once (0: none; sizes above 8 are allowed first), cached per
// (device, kernel, size).
static int cluster_capacity(const void *fn, int size, int threads) {
    struct Entry {
        int dev;
        const void *fn;
        int size;
        int n;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].size == size) return cache[i].n;
    int clusters = 0;
    if (size <= 8 || cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                         cudaSuccess) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)size;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)size);
        cfg.blockDim = dim3((unsigned)threads);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) clusters = 0;
    }
    cudaGetLastError();  // a refused query leaves no error behind
    if (ncache < 32) cache[ncache++] = Entry{dev, fn, size, clusters};
    return clusters;
}

template <typename T, bool VEC>
static cudaError_t launch_chain_t(ChainArgs a, VocabPlan p, WsView w, cudaStream_t st) {
    void *args[] = {&a, &p, &w};
    const unsigned items = (unsigned)((size_t)a.B * p.rows_per_seq * p.nchunks);
    cudaError_t e;
    if constexpr (VEC) {
        // streaming form: one CTA per SM (fewer when there are fewer units)
        const void *fn = (const void *)chain_stats_stream_kernel<T>;
        const int smem = kSStages * kSUnitBytes;
        static int attr_set[64] = {0};
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if (dev < 64 && !attr_set[dev]) {
            if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                cudaSuccess)
                return e;
            attr_set[dev] = 1;
        }
        int sms = device_sm_count();
        if (sms <= 0) return cudaErrorUnknown;
        if (p.max_ctas > 0 && p.max_ctas < sms) sms = p.max_ctas;
        const unsigned grid = (unsigned)(items < (unsigned)sms ? items : (unsigned)sms);
        e = launch_pdl(fn, dim3(grid), dim3(kSThreads), smem, st, args);
    } else {
        e = launch_pdl((const void *)chain_stats_kernel<T, VEC>, dim3(items), dim3(kVT), 0, st,
                       args);
    }
    if (e != cudaSuccess) return e;
    const unsigned res = (unsigned)((size_t)a.B * p.res_chunks);
    if constexpr (VEC) {
        // The whole GPU: a cluster per sequence, while the sequences take at
        // most 7/8 of the clusters the device holds at once.  Nearer the
        // limit (B = 30 and 32 sequences of 16 chunks, against 33 clusters on
        // 152 SMs) some clusters found no room until others had left, and the
        // call ran 1.5-2.3 us longer than with the counted form; at 28 it ran
        // 2.6 us shorter.
        const void *cfn = (const void *)chain_residual_kernel<T, VEC, true>;
        if (p.max_ctas == 0 && p.res_chunks <= kMaxResCluster &&
            (long long)a.B * 8 <= (long long)cluster_capacity(cfn, p.res_chunks, kVT) * 7) {
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)p.res_chunks;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(res);
            cfg.blockDim = dim3(kVT);
            cfg.dynamicSmemBytes = 0;
            cfg.stream = st;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            return cudaLaunchKernelExC(&cfg, cfn, args);
        }
    }
    return launch_pdl((const void *)chain_residual_kernel<T, VEC, false>, dim3(res), dim3(kVT), 0,
                      st, args);
}

template <typename T, bool VEC>
static cudaError_t launch_tree_t(TreeArgs a, VocabPlan p, WsView w, cudaStream_t st) {
    void *args[] = {&a, &p, &w};
    const unsigned items = (unsigned)((size_t)a.B * p.rows_per_seq * p.nchunks);
    if constexpr (VEC) {
        // streaming argmax pass (one CTA per SM, fewer for fewer units), then the walk
        const void *fn = (const void *)tree_stats_stream_kernel<T>;
        const int smem = kSStages * kSUnitBytes;
        static int attr_set[64] = {0};
        int dev = 0;
        cudaError_t e;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if (dev < 64 && !attr_set[dev]) {
            if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                cudaSuccess)
                return e;
            attr_set[dev] = 1;
        }
        int sms = device_sm_count();
        if (sms <= 0) return cudaErrorUnknown;
        if (p.max_ctas > 0 && p.max_ctas < sms) sms = p.max_ctas;
        const unsigned grid = (unsigned)(items < (unsigned)sms ? items : (unsigned)sms);
        if ((e = launch_pdl(fn, dim3(grid), dim3(kSThreads), smem, st, args)) != cudaSuccess) return e;
        return launch_pdl((const void *)tree_decide_kernel<T>, dim3((unsigned)a.B), dim3(kVT), 0, st,
                          args);
    } else {
        return launch_pdl((const void *)tree_stats_kernel<T, VEC>, dim3(items), dim3(kVT), 0, st,
                          args);
    }
}

sv_status launch_verify_chain(const ChainArgs &a, int dtype, const VocabPlan &p, void *ws,
                              cudaStream_t st) {
    if (a.N > kMaxChainN || p.res_chunks > kMaxResChunks) return SV_ERR_UNSUPPORTED;
    const WsView w = ws_view(ws, p, a.B);
    cudaError_t e;
    if (dtype == SV_BF16)
        e = p.vec ? launch_chain_t<uint16_t, true>(a, p, w, st)
                  : launch_chain_t<uint16_t, false>(a, p, w, st);
    else
        e = p.vec ? launch_chain_t<float, true>(a, p, w, st)
                  : launch_chain_t<float, false>(a, p, w, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status launch_verify_tree_greedy(const TreeArgs &a, int dtype, const VocabPlan &p, void *ws,
                                    cudaStream_t st) {
    if (a.T > kMaxTreeT) return SV_ERR_UNSUPPORTED;
    const WsView w = ws_view(ws, p, a.B);
    cudaError_t e;
    if (dtype == SV_BF16)
        e = p.vec ? launch_tree_t<uint16_t, true>(a, p, w, st)
                  : launch_tree_t<uint16_t, false>(a, p, w, st);
    else
        e = p.vec ? launch_tree_t<float, true>(a, p, w, st)
                  : launch_tree_t<float, false>(a, p, w, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

namespace sv {

VocabPlan plan_vocab_stree(int B, int T, int V, int dtype) {
    VocabPlan p{};
    const int esz = dtype == SV_F32 ? 4 : 2;
    const int per_vec = 16 / esz;
    p.rows_per_seq = 2 * T;
    p.chunk_elems = kVT * kLoadsPerThread * per_vec;
    p.nchunks = (V + p.chunk_elems - 1) / p.chunk_elems;
    p.vec = ((size_t)V * esz) % 16 == 0;
    p.recs_per_unit = 1;
    p.off_counters = 0;
    p.off_partials = 0;
    p.bytes = align_up(sizeof(float2) * (size_t)B * p.rows_per_seq * p.nchunks, 256);
    return p;
}

// Largest cluster the device schedules for the walk: 16 CTAs (a non-portable
// size) where it can run one, else the portable 8.  Queried once per device
// and kernel.
static int walk_cluster_max(const void *fn) {
    return cluster_capacity(fn, kWClusterMax, kWT) > 0 ? kWClusterMax : 8;
}

template <typename T, bool VEC>
static cudaError_t launch_stree_t(STreeArgs a, VocabPlan p, float2 *rec, cudaStream_t st) {
    void *args[] = {&a, &p, &rec};
    const unsigned items = (unsigned)((size_t)a.B * p.rows_per_seq * p.nchunks);
    cudaError_t e = launch_pdl((const void *)stree_stats_kernel<T, VEC>, dim3(items), dim3(kVT), 0,
                               st, args);
    if (e != cudaSuccess) return e;
    // the walk: one cluster per sequence, launched after the statistics pass has
    // finished (a cluster placed early, beside that pass, can wait long for SMs)
    const void *wfn = (const void *)stree_walk_kernel<T, VEC>;
    const int C = walk_cluster_max(wfn);
    if (C < 1) return cudaErrorUnknown;
    p.walk_cluster = C;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * C));
    cfg.blockDim = dim3(kWT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, wfn, args);
}

sv_status launch_verify_tree_stochastic(const STreeArgs &a, int dtype, const VocabPlan &p, void *ws,
                                        cudaStream_t st) {
    if (a.T > kMaxTreeT || (a.V + 8 * kWT - 1) / (8 * kWT) > kMaxWSeg) return SV_ERR_UNSUPPORTED;
    float2 *rec = static_cast<float2 *>(ws);
    cudaError_t e;
    if (dtype == SV_BF16)
        e = p.vec ? launch_stree_t<uint16_t, true>(a, p, rec, st)
                  : launch_stree_t<uint16_t, false>(a, p, rec, st);
    else
        e = p.vec ? launch_stree_t<float, true>(a, p, rec, st)
                  : launch_stree_t<float, false>(a, p, rec, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

#ifdef SV_PHASE_STAMPS
// Spans of the kernels above (first start, last end; globaltimer ns), in the
// order chain statistics, chain residual draw, tree argmax pass, tree walk.
extern "C" int sv_debug_vocab_spans(unsigned long long *dst) {
    return cudaMemcpyFromSymbol(dst, sv::g_vspan, sizeof(sv::g_vspan)) == cudaSuccess ? 0 : -1;
}
extern "C" int sv_debug_vocab_clear(void) {
    unsigned long long init[sv::kSpanCount][2];
    for (int i = 0; i < sv::kSpanCount; ++i) {
        init[i][0] = ~0ull;
        init[i][1] = 0ull;
    }
    return cudaMemcpyToSymbol(sv::g_vspan, init, sizeof(init)) == cudaSuccess ? 0 : -1;
}
#endif
