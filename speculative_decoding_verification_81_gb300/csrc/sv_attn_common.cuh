// sv_attn_common.cuh -- pieces shared by the attention kernels: tile
// geometry, kernel parameters, the balanced split of (sequence, KV head, row
// group, tile) units over persistent CTAs, and the per-call prologue.
#pragma once

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kD = 128;
constexpr int kBK = 128;                  // keys per tile
constexpr int kBox = kBK * 64 * 2;        // one 128-key x 64-dim bf16 TMA box: 16 KB
constexpr int kStageBytes = 4 * kBox;     // K lo/hi + V lo/hi: 64 KB
constexpr int kMaxB = 4096;
constexpr int kMinPage = 8;                      // smallest page (a swizzle atom of rows)
constexpr int kMaxSubBlocks = kBK / kMinPage;    // pages per key tile at most
constexpr int kMaxT = 64;
constexpr int kMinTilesPerCta = 8;  // key tiles a CTA takes at least (small problems)
constexpr int kMaxCluster = 8;      // CTAs of a cluster in cluster mode (a portable size)
constexpr int kSoftmaxWarps = 8;                      // warps 2-9: two per TMEM lane quarter
constexpr int kPvWarp = 2 + kSoftmaxWarps;              // issues the PV products
constexpr int kVLoadWarp = 3 + kSoftmaxWarps;           // loads the V tiles
constexpr int kTcThreads = 32 * (4 + kSoftmaxWarps);    // + K-load and S-issue warps

struct AttnKParams {
    const uint16_t *q;
    uint16_t *out;
    const int32_t *prefix_lens;
    const int32_t *parents;
    int32_t *seq_status;
    int B, T, Hq, Hkv, G, S_max, M, RG, rows_per_rg;
    float scale_log2;
    float *part_o;   // [grid][2][kD / 4][MROWS] float4 (chunk-major): unnormalised O of split pairs
    float *part_ml;  // [grid][2][rows_per_rg][2 halves][2]: (max in log2 units, row sum)
    int *pair_ctr;   // [B][Hkv][RG][2][8]: per softmax warp, CTAs arrived / partials ready (0 after the merge)
    // paged caches (block_table non-null): K/V [num_pages][Hkv][page_size][D];
    // logical slot s of sequence b is in page block_table[b][s / page_size]
    const int32_t *block_table;
    int max_pages, num_pages, page_size;
    // per-sequence node counts T_b (1 <= T_b <= T; nodes past T_b are padding), or null: all T
    const int32_t *node_counts;
    // cluster mode (cluster > 1): one thread-block cluster of `cluster` CTAs per
    // (sequence, KV head, row group), CTA k of it taking the k-th contiguous
    // share of that group's key tiles; the shares are merged in distributed
    // shared memory.  0 or 1: the flat split over persistent CTAs.
    int cluster;
    int node_count_add;  // T_b = node_counts[b] + node_count_add
    // fused tree step in cluster mode (hook.step_ctr null otherwise): after a
    // cluster's group is read, it arrives on its (sequence, KV head) counter;
    // the last arrival moves the accepted path's rows (hook_acc, hook_path:
    // the walk's outputs, path rows hook_path_stride apart)
    StepHook hook;
    const int32_t *hook_acc;
    const int32_t *hook_path;
    int hook_path_stride;
};

// Position in the unit list: sequence, (kv head * RG + row group), tile.
// Position in a CTA's run of units (sequence, pair, tile): the pairs a run
// visits are pr = pi * pstride + poff for pi = 0..npr-1 (all pairs, or one row
// group of every KV head).
struct Cursor {
    int b, pr, tile, n, pi;
};

__device__ __forceinline__ long long cta_begin(long long U, int grid, int c) {
    return (U * c) / grid;
}

// Index of the CTA whose range holds unit u.
__device__ __forceinline__ int cta_of(long long U, int grid, long long u) {
    return (int)(((u + 1) * grid + U - 1) / U) - 1;
}

// Pairs a CTA's run visits: npr per sequence, pair pi is pr = pi * pstride + poff.
struct PairLane {
    int npr, pstride, poff;
};

__device__ __forceinline__ Cursor cursor_at(const int *tile_base, int B, PairLane pl, long long u) {
    int lo = 0, hi = B - 1;  // last b with tile_base[b] * npr <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)tile_base[mid] * pl.npr <= u) lo = mid;
        else hi = mid - 1;
    }
    Cursor c;
    c.b = lo;
    c.n = tile_base[lo + 1] - tile_base[lo];
    const long long rem = u - (long long)tile_base[lo] * pl.npr;
    c.pi = c.n > 0 ? (int)(rem / c.n) : 0;
    c.pr = c.pi * pl.pstride + pl.poff;
    c.tile = c.n > 0 ? (int)(rem - (long long)c.pi * c.n) : 0;
    return c;
}

__device__ __forceinline__ void cursor_next(Cursor &c, const int *tile_base, int B, PairLane pl) {
    if (++c.tile < c.n) return;
    c.tile = 0;
    if (++c.pi < pl.npr) {
        c.pr = c.pi * pl.pstride + pl.poff;
        return;
    }
    c.pi = 0;
    c.pr = pl.poff;
    do {
        ++c.b;
    } while (c.b < B && tile_base[c.b + 1] == tile_base[c.b]);
    c.n = c.b < B ? tile_base[c.b + 1] - tile_base[c.b] : 0;
}

// Barrier of several warps on an mbarrier counting one arrival per warp
// (bounded, unlike bar.sync); the verdict is the same in every lane.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &uses) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = warp_wait_bounded(bar, uses & 1);
    ++uses;
    return ok;
}

// The tile row maxima of the two softmax warps of a lane quarter, exchanged
// through one 64-bit word per lane: the value's bits with the tile's tag
// (tile counter + 1) above them, stored and polled with volatile shared
// accesses.  A naturally aligned 64-bit access is seen whole, so the tag
// that matches also vouches for the value, and no barrier or fence is needed.
__device__ __forceinline__ void xchg_put(uint64_t *slot, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
    asm volatile("st.volatile.shared.u64 [%0], %1;" ::"r"(smem_u32(slot)), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t xchg_peek(const uint64_t *slot) {
    uint64_t w;
    asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(w) : "r"(smem_u32(slot)) : "memory");
    return w;
}

// The partner's value for the tile `tag`, by a whole warp (one verdict for
// all lanes); false after kWaitCycles.
__device__ __forceinline__ bool xchg_get(const uint64_t *slot, uint32_t tag, float &v) {
    uint64_t w = xchg_peek(slot);
    if (!__all_sync(0xffffffffu, (uint32_t)(w >> 32) == tag)) {
        const long long t0 = clock64();
        while (true) {
            w = xchg_peek(slot);
            if (__all_sync(0xffffffffu, (uint32_t)(w >> 32) == tag)) break;
            if (__any_sync(0xffffffffu, clock64() - t0 > kWaitCycles)) return false;
        }
    }
    v = __uint_as_float((uint32_t)w);
    return true;
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// The running row max only moves when a tile's max exceeds it by more than
// this many log2 units; until then probabilities stay below 2^8 relative to
// the stale max, which the f32 sums and the bf16 P carry without loss, and
// the final division by the row sum is unchanged.
constexpr float kRescaleThreshold = 8.0f;

// Every CTA: tiles per sequence and their prefix sums into tile_base[0..B]
// (identically in every CTA); CTA 0 also writes each sequence's status
// (prefix length in range, parent array a topologically ordered tree).
// Contains __syncthreads: call from every thread of the CTA.
// Nodes of sequence b: T_b, or 0 when out of range (the sequence is then invalid).
__device__ __forceinline__ int nodes_of(const AttnKParams &p, int b) {
    if (!p.node_counts) return p.T;
    const int n = p.node_counts[b] + p.node_count_add;
    return (n >= 1 && n <= p.T) ? n : 0;
}

// Every sequence's inputs checked and its status written, by CTA 0 (out of
// line: the other CTAs jump over one call instead of the whole check).
static __device__ __noinline__ void check_sequences(const AttnKParams &p, int nt) {
    const int tid = threadIdx.x;
    for (int b = tid; b < p.B; b += nt) {
        const int L = p.prefix_lens[b], Tb = nodes_of(p, b);
        bool ok = L >= 0 && Tb > 0 && (long long)L + Tb <= p.S_max;
        if (ok && p.block_table) {  // the pages holding slots [0, L + T_b) exist
            const int np = (L + Tb + p.page_size - 1) / p.page_size;
            for (int j = 0; j < np; ++j) {
                const int pg = p.block_table[(size_t)b * p.max_pages + j];
                if (pg < 0 || pg >= p.num_pages) ok = false;
            }
        }
        p.seq_status[b] = ok ? SV_OK : SV_ERR_BAD_INPUT;
    }
    __syncthreads();
    if (p.parents) {
        for (int i = tid; i < p.B * p.T; i += nt) {
            const int b = i / p.T, t = i - b * p.T;
            if (t >= nodes_of(p, b)) continue;  // padding node
            const int pa = p.parents[i];
            if (t == 0 ? pa != -1 : (pa < 0 || pa >= t)) p.seq_status[b] = SV_ERR_BAD_INPUT;
        }
    }
}

// pre_L, pre_T: prefix length and node count of sequence threadIdx.x, loaded
// by the caller ahead of its own set-up.
__device__ __forceinline__ void attn_prologue(const AttnKParams &p, int *tile_base, int nt, int pre_L,
                                              int pre_T) {
    const int tid = threadIdx.x;
    for (int b = tid; b < p.B; b += nt) {
        const int L = b == tid ? pre_L : p.prefix_lens[b];
        const int Tb = b == tid ? pre_T : nodes_of(p, b);
        const bool ok = L >= 0 && Tb > 0 && (long long)L + Tb <= p.S_max;
        tile_base[b] = ok ? (L + Tb + kBK - 1) / kBK : 0;
    }
    __syncthreads();
    if (tid < 32) {  // exclusive scan, 32 sequences at a time
        int carry = 0;
        for (int c0 = 0; c0 < p.B; c0 += 32) {
            const int b = c0 + tid;
            const int v = b < p.B ? tile_base[b] : 0;
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (tid >= off) x += y;
            }
            if (b < p.B) tile_base[b] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (tid == 0) tile_base[p.B] = carry;
    }
    if (blockIdx.x == 0 && p.seq_status) check_sequences(p, nt);
    __syncthreads();
}

// Ancestor set of node t (bit j = node j on the root->t path) from sequence
// b's parent array held across a warp (lane l has the parents of nodes l and
// 32 + l, -1 past T): the path is walked with shuffles, not dependent loads.
// At most 64 steps; a parent that does not precede its child ends the walk
// (the call reports such a tree as bad).  Every lane of the warp calls it; a
// lane with valid == false gets 0.  chain (parents NULL): the causal set.
__device__ __forceinline__ uint64_t ancestors_warp(bool chain, int par_lo, int par_hi, int t,
                                                   bool valid) {
    if (chain) return !valid ? 0ull : t >= 63 ? ~0ull : ((1ull << (t + 1)) - 1ull);
    uint64_t anc = 0;
    int nd = valid ? t : -1;
    for (int step = 0; step < kMaxT; ++step) {
        if (__all_sync(0xffffffffu, nd < 0)) break;
        if (nd >= 0) anc |= 1ull << nd;
        const int lo = __shfl_sync(0xffffffffu, par_lo, nd & 31);
        const int hi = __shfl_sync(0xffffffffu, par_hi, nd & 31);
        const int pn = nd >= 32 ? hi : lo;
        if (nd >= 0) nd = pn < nd ? pn : -1;  // up to the root; a parent not before its node ends it
    }
    return anc;
}

// Parents of nodes lane and 32 + lane of sequence b (-1 past T or for a chain).
__device__ __forceinline__ int2 load_parents_warp(const int32_t *parents, int T, int b, int lane) {
    if (!parents) return make_int2(-1, -1);
    const int32_t *row = parents + (size_t)b * T;
    return make_int2(lane < T ? row[lane] : -1, 32 + lane < T ? row[32 + lane] : -1);
}

}  // namespace sv
