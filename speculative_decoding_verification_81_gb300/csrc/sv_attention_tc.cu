// sv_attention_tc.cu -- verification attention on the 5th-generation tensor
// cores (tcgen05), accumulators in tensor memory.
//
// Source: "Chapitre 9 -- Décodage spéculatif" §9.1 (one forward over the
// prefix concatenated with the candidates; the pass stays memory-bound) and
// §9.2 (EAGLE-2 draft tree verified in one attention pass with a custom
// mask); "Parallel Decoding" glossary, Medusa "Tree attention" and
// "L'attention en arbre : la brique commune".
//
// The G = Hq/Hkv query heads of a KV head and the T nodes form M = G*T query
// rows that share every K/V tile, so each tile is read from HBM once per
// (sequence, KV head) and feeds up to 128 rows of tensor-core work.  Work is
// the flat list of (sequence, KV head, 128-row group, 128-key tile) units; a
// persistent grid (one CTA per SM) takes equal contiguous ranges of it, so the
// load is balanced whatever the prefix lengths.  A (sequence, KV head) whose
// tiles fall to several CTAs is merged by the CTA that finishes its part
// last: it combines the others' partials (O, max, sum) with its own O.
// Small problems (few row groups: the Medusa tree, short batches) run in
// cluster mode instead: one thread-block cluster per row group, its CTAs
// taking contiguous shares of the group's tiles, the shares exchanged
// through L2 after one cluster barrier, each CTA finishing a slice of the
// rows.  Inside a CTA (12 warps):
//
//   warps 0, 11 TMA producers: K and V tiles (2-D tensor maps, 128-byte
//               swizzle) into a ring of STAGES shared-memory stages, K and
//               V halves refilled independently (K as soon as its S product
//               is done, V after its PV).
//   warp 1      owns the tensor memory (512 columns); one lane issues the
//               S = Q K^T products (M=128 or 64 rows, N=128 keys, K=128)
//               into one of three TMEM S buffers (columns 0-383; O at
//               384-511), so that S of tile j + 2 is computed while tile j's
//               P waits for its PV product.
//   warp 10     one lane issues O += P V (N=128, K=128 keys) into the TMEM
//               O accumulator.  P is read from TMEM; Q, K (K-major) and V
//               (MN-major) from shared memory (Q from its own double buffer).  The
//               tiles are 128 keys wide because a product's issue and
//               completion take about the same time for small and large
//               shapes: fewer, larger MMAs keep the tensor pipe fed.
//   warps 2-9   softmax, two threads per query row: a warp may only touch
//               the TMEM lane quarter of its SM sub-partition (warp % 4), so
//               warps w and w+4 share the rows of one quarter, the first
//               taking keys (and output columns) 0-63 of every tile, the
//               second 64-127.  Each reads its half S row from TMEM, applies
//               the ancestor mask (a 64-bit set of tree ancestors per row,
//               only in the tile(s) holding the T new rows), agrees the tile
//               max with its partner through a tagged shared-memory word per
//               lane (value and tile number in one 64-bit store, polled by
//               the partner, no barrier), keeps the running
//               max (moved only when it grows by more than 2^8, its half of
//               the O row then rescaled in TMEM) and its part of the row sum,
//               writes its bf16 P half row over the S columns it came from
//               (the A operand of the PV MMA), and at the end of a segment
//               reads its half of the O row and writes it out (or a partial).
//               The loop runs segment by segment: the tiles between a
//               segment's first one and those holding new rows take a short
//               form of the tile code, without those per-tile checks.
//
// The two issuing lanes wait (blocking, bounded) on their own barriers, so S
// of the next tile is issued while the softmax of the current one runs, PV
// of a tile the moment its P is written, and no K/V stage is held longer
// than its own tile needs.  Every wait is bounded (SV_ERR_TIMEOUT on expiry);
// the TMEM is always released.
#include <type_traits>

#include "sv_attn_common.cuh"
#include "sv_internal.h"

namespace sv {

// Tensor-memory columns (32-bit each, one row per lane): three S buffers
// (128 f32 each; the bf16 P of keys 0-63 overwrites S columns 0-31, that of
// keys 64-127 S columns 64-95) and the O accumulator (128 f32).  P is the A
// operand of the PV product, read by the tensor core from TMEM; Q, the A
// operand of S, sits in shared memory (double-buffered, loaded by TMA ahead
// of its segment).
constexpr uint32_t kTcCols = 512;

// Phase stamps (a diagnostic build only, -DSV_PHASE_STAMPS): the SM clock at
// fixed points of every CTA's run (slot 0: the globaltimer at entry, slot 1
// the clock there, to place the CTAs on one time line), read back by
// sv_debug_attention_stamps.  The library proper compiles them out.
#ifdef SV_PHASE_STAMPS
constexpr int kStampSlots = 32;
constexpr int kStampCtas = 1024;
static __device__ long long g_stamps[kStampCtas * kStampSlots];
__device__ __forceinline__ void phase_stamp(int slot, long long value) {
    if (blockIdx.x < kStampCtas) g_stamps[blockIdx.x * kStampSlots + slot] = value;
}
__device__ __forceinline__ long long sm_id() {
    unsigned r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}
__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#define SV_STAMP(slot) phase_stamp((slot), clock64())
#define SV_STAMP_ENTRY()                \
    do {                                \
        phase_stamp(1, clock64());      \
        phase_stamp(0, global_ns());    \
        phase_stamp(23, sm_id());       \
    } while (0)
#define SV_STAMP_VALUE(slot, v) phase_stamp((slot), (long long)(v))
// slot 22: the clock at the exit of the CTA's last warp (every warp, at every exit)
struct StampExit {
    __device__ ~StampExit() {
        if ((threadIdx.x & 31) == 0 && blockIdx.x < kStampCtas)
            atomicMax(reinterpret_cast<unsigned long long *>(&g_stamps[blockIdx.x * kStampSlots + 22]),
                      (unsigned long long)clock64());
    }
};
#define SV_STAMP_EXIT() StampExit sv_stamp_exit_
#else
#define SV_STAMP_EXIT() ((void)0)
#define SV_STAMP(slot) ((void)0)
#define SV_STAMP_ENTRY() ((void)0)
#define SV_STAMP_VALUE(slot, v) ((void)0)
#endif
// S buffers in tensor memory: with three, S of tile j + 2 is computed while
// tile j's P waits for its PV product (with two, the softmax waited ~0.1 us a
// tile for S on 128-row groups)
constexpr int kSBufs = 3;
constexpr uint32_t kColS = 0, kColO = kSBufs * 128;

// Byte offset of 16-byte chunk c (0..7) of row `row` in a 128-byte-swizzled
// block whose rows are 128 bytes (the layout TMA writes with SWIZZLE_128B and
// the tensor core reads with swizzle mode 2).  Used to zero V rows.
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4));
}

struct TcSmem {
    uint64_t full_k[4], empty_k[4];  // TMA ring, K halves of the stages
    uint64_t full_v[4], empty_v[4];  // V halves
    uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];  // per S buffer
    uint64_t q_full[2], q_empty[2];  // Q tiles in shared memory (double buffer)
    uint64_t fin, fin_pv;
    uint64_t pair[4];            // the two softmax warps of each lane quarter, at segment ends
    uint64_t k_first;            // the first K tile has been requested
    uint64_t xmax[2][4][2][32];  // [tile parity][quarter][half][lane]: half-row tile maxima, tagged
    float xl[4][2][32];          // [quarter][half][lane]: half-row sums at a segment end
    uint32_t tmem;
    int abort_flag;
    int hook_last;  // fused step: this cluster brought its counter to the end
};

// ---------------------------------------------------------------- cluster mode
//
// The CTAs of a cluster each hold an unnormalised share (O, max, sum) of every
// row of the group; CTA k finishes rows k*MROWS/cs .. (its "own" rows).  Each
// CTA writes its share to its slot of the workspace (the flat mode's partial
// slots), the cluster meets at a barrier (release/acquire: the writes are
// visible after it), and each CTA reads the shares of its own rows back from
// L2.  In a slot, O is stored chunk-major -- 16-byte chunk c (columns 4c..4c+3)
// of row r at (c * MROWS + r) * 16 bytes -- so that the lanes of a warp, one
// row each, write and read consecutive 16 bytes; the (max, sum) pairs follow
// at float offset MROWS * kD, one per row.  (Shares sent through distributed
// shared memory -- per-thread loads, or one bulk copy per owner -- took
// longer on the Medusa-tree shape: about 1.5 us against 0.7.)

// Floats of a CTA's share: O (MROWS x kD) then the (max, sum) pairs; it fits
// in the CTA's flat-mode partial region of 2 * MROWS * kD floats.
template <int MROWS>
constexpr size_t kClusterSlot = (size_t)MROWS * kD + 2 * MROWS;
static_assert(kClusterSlot<128> <= 2 * 128 * kD && kClusterSlot<64> <= 2 * 64 * kD,
              "cluster share larger than the partial slot");

// A softmax thread's half row of O (64 columns at TMEM address o_half) and,
// from the first half's thread, the row's (max, sum), into this CTA's share
// `slot`.  Warp-collective (TMEM loads): every lane calls it; has_row: the
// lane owns row r (with 64-row groups, lanes 16-31 own none).
template <int MROWS>
__device__ __forceinline__ void cluster_stage(float *slot, uint32_t o_half, int r, int half,
                                              bool has_row, bool row_valid, float m, float lrow) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t ov[32];
        __syncwarp();
        tc::tmem_ld32(o_half + 32 * h, ov);
        tc::wait_ld();
        if (!row_valid) continue;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            __stcg(reinterpret_cast<float4 *>(slot) + (size_t)(half * 16 + h * 8 + c) * MROWS + r,
                   make_float4(__uint_as_float(ov[4 * c]), __uint_as_float(ov[4 * c + 1]),
                               __uint_as_float(ov[4 * c + 2]), __uint_as_float(ov[4 * c + 3])));
    }
    if (half == 0 && has_row)
        __stcg(reinterpret_cast<float2 *>(slot + MROWS * kD) + r,
               row_valid ? make_float2(m, lrow) : make_float2(kNegInf, 0.f));
}

// Rows crank*MROWS/CS .. of the cluster's group from the CS shares (CTA i of
// the cluster: its slot at slot0 + i * slot_stride floats): weights
// 2^(m_i - max m), the weighted O rows summed in rank order and divided by the
// weighted row sums; bf16 out.  Thread t256 of the 256 softmax threads takes
// row t256 % rows and the chunks t256 / rows + j * (256 / rows): a warp reads
// one chunk of consecutive rows.
template <int MROWS, int CS>
__device__ __forceinline__ void cluster_merge_cs(const AttnKParams &p, const float *slot0,
                                                 size_t slot_stride, int crank, int b, int kvh,
                                                 int rg, int ntiles, int t256) {
    constexpr int kRpc = MROWS / CS;                 // rows this CTA finishes
    constexpr int kGroups = kSoftmaxWarps * 32 / kRpc;  // chunk groups: threads per row
    constexpr int kChunks = 32 / kGroups;            // 16-byte chunks (4 columns) per thread
    static_assert(kGroups <= 32 && kChunks >= 1, "cluster too large for the row group");
    const int lr = t256 % kRpc, cg = t256 / kRpc;
    const int r = crank * kRpc + lr;
    const int rglob = rg * p.rows_per_rg + r;
    if (b >= p.B || ntiles <= 0 || r >= p.rows_per_rg || rglob >= p.M) return;
    const int t = rglob / p.G, g = rglob - t * p.G;
    if (t >= nodes_of(p, b)) return;
    // every share's (max, sum) and O chunks in flight at once
    float2 ml[CS];
    float4 o[kChunks][CS];
#pragma unroll
    for (int i = 0; i < CS; ++i) {
        const float *sl = slot0 + i * slot_stride;
        ml[i] = __ldcg(reinterpret_cast<const float2 *>(sl + MROWS * kD) + r);
#pragma unroll
        for (int j = 0; j < kChunks; ++j)
            o[j][i] = __ldcg(reinterpret_cast<const float4 *>(sl) + (size_t)(cg + j * kGroups) * MROWS + r);
    }
    float ms = kNegInf;
#pragma unroll
    for (int i = 0; i < CS; ++i) ms = fmaxf(ms, ml[i].x);
    float w[CS], lsum = 0.f;
#pragma unroll
    for (int i = 0; i < CS; ++i) {
        w[i] = ml[i].x == kNegInf ? 0.f : ex2_approx(ml[i].x - ms);  // an empty share weighs 0
        lsum = __fmaf_rn(ml[i].y, w[i], lsum);
    }
    const float inv = 1.f / lsum;
    uint16_t *orow = p.out + (((size_t)b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < CS; ++i) {
            // an empty share's slot holds no O: select, never multiply, it
            const bool use = w[i] != 0.f;
            acc.x = use ? __fmaf_rn(o[j][i].x, w[i], acc.x) : acc.x;
            acc.y = use ? __fmaf_rn(o[j][i].y, w[i], acc.y) : acc.y;
            acc.z = use ? __fmaf_rn(o[j][i].z, w[i], acc.z) : acc.z;
            acc.w = use ? __fmaf_rn(o[j][i].w, w[i], acc.w) : acc.w;
        }
        *reinterpret_cast<uint2 *>(orow + 4 * (cg + j * kGroups)) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
}

template <int MROWS>
__device__ __forceinline__ void cluster_merge(const AttnKParams &p, const float *slot0,
                                              size_t slot_stride, int cs, int crank, int b,
                                              int kvh, int rg, int ntiles, int t256) {
    if (cs == 2) cluster_merge_cs<MROWS, 2>(p, slot0, slot_stride, crank, b, kvh, rg, ntiles, t256);
    else if (cs == 4) cluster_merge_cs<MROWS, 4>(p, slot0, slot_stride, crank, b, kvh, rg, ntiles, t256);
    else cluster_merge_cs<MROWS, 8>(p, slot0, slot_stride, crank, b, kvh, rg, ntiles, t256);
}

// Compaction of one (sequence, KV head) in a fused tree step, by the 128
// threads of the producer and MMA warps (t128), idle once the cluster barrier
// is passed: rows L + path[d] -> L + d for d = 1..a, K and V.  Every source
// row goes to shared memory (the idle K/V ring) before any row is written,
// so an in-place move never reads a row another move has overwritten.
// bar_id: a named barrier over exactly these 128 threads.
__device__ __forceinline__ void hook_move_rows(const AttnKParams &p, int b, int kvh, uint4 *bounce,
                                               int t128, int bar_id) {
    const int a = __ldcg(p.hook_acc + b);
    const int L = __ldcg(p.hook.prefix_lens + b);
    const int Tb = nodes_of(p, b);
    // a < 0: the sequence's tree or tokens were invalid; a cache that cannot
    // hold the nodes: nothing was read for it either way
    if (a <= 0 || L < 0 || Tb <= 0 || (long long)L + Tb > p.S_max || a >= Tb) return;
    const int32_t *path = p.hook_path + (size_t)b * p.hook_path_stride;
    constexpr int kWords = kD * 2 / 16;  // 16-byte words of a row
    const size_t head = ((size_t)b * p.Hkv + kvh) * p.S_max;
    const int n = a * 2 * kWords;
    for (int w = t128; w < n; w += 128) {
        const int d = 1 + w / (2 * kWords), kv = (w / kWords) & 1, word = w % kWords;
        int src = __ldcg(path + d);
        if (src < d || src >= Tb) src = d;  // (a walk's path never does this; stay in the sequence's rows)
        const uint4 *from = kv ? p.hook.v : p.hook.k;
        bounce[w] = from[(head + L + src) * kWords + word];
    }
    __syncwarp();
    named_bar_sync(bar_id, 128);
    for (int w = t128; w < n; w += 128) {
        const int d = 1 + w / (2 * kWords), kv = (w / kWords) & 1, word = w % kWords;
        if (__ldcg(path + d) == d) continue;  // already in place
        uint4 *to = kv ? p.hook.v : p.hook.k;
        to[(head + L + d) * kWords + word] = bounce[w];
    }
}

template <int MROWS>
__device__ __forceinline__ void cluster_merge(const AttnKParams &p, const float *o_base,
                                              size_t o_stride, const float *ml_base,
                                              size_t ml_stride, int cs, int crank, int b, int kvh,
                                              int rg, int ntiles, int t256) {
    if (cs == 2)
        cluster_merge_cs<MROWS, 2>(p, o_base, o_stride, ml_base, ml_stride, crank, b, kvh, rg, ntiles, t256);
    else if (cs == 4)
        cluster_merge_cs<MROWS, 4>(p, o_base, o_stride, ml_base, ml_stride, crank, b, kvh, rg, ntiles, t256);
    else
        cluster_merge_cs<MROWS, 8>(p, o_base, o_stride, ml_base, ml_stride, crank, b, kvh, rg, ntiles, t256);
}

// Out-of-line pieces of the softmax warps' per-tile loop (each runs at most
// once a segment or when the running max moves), so that the loop's own code
// stays short: inline, the code it jumps over cost instruction fetch stalls
// every tile (the softmax of 128-row groups paced ~6% slower).

// Once the PV product behind `bar` is done: this warp's 64 O columns from
// TMEM address o_cols times a.  False when the wait gave up (the columns are
// scaled anyway; the caller reports the failure).
__device__ __noinline__ bool rescale_o_half(uint64_t *bar, uint32_t parity, uint32_t o_cols, float a) {
    const bool ok = warp_wait_bounded(bar, parity);
    tc::fence_after();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t ov[32];
        tc::tmem_ld32(o_cols + 32 * h, ov);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * a);
        tc::tmem_st32(o_cols + 32 * h, ov);
    }
    return ok;
}

// Once the V half behind `bar` has landed: its rows z0 .. kBK - 1 (past the
// sequence's last slot) zeroed in shared memory at vst, by the softmax
// threads (t: 0 .. 32 * kSoftmaxWarps - 1), visible to the tensor core.
// False when the wait gave up.
__device__ __noinline__ bool zero_v_tail(uint64_t *bar, uint32_t parity, uint8_t *vst, int z0, int t) {
    if (!warp_wait_bounded(bar, parity)) return false;
    for (int i = t; i < (kBK - z0) * 16; i += 32 * kSoftmaxWarps) {
        const int row = z0 + (i >> 4), c = i & 15;
        *reinterpret_cast<uint4 *>(vst + (c >> 3) * kBox + sw128(row, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
    return true;
}

// The end of a segment for one softmax warp: its rows' sum from the column
// halves, then this half of the O rows out of TMEM -- written out (whole
// segment, or the merging CTA of a split pair), left as a partial, or staged
// for the cluster merge.  Kept out of line: it runs once a segment, and the
// per-tile loop stays short.  Returns the warp's updated pair-barrier count,
// the partial counter to flag ready after the next tile (or null) and whether
// the rows were staged; ok is false when a bounded wait gave up.
struct SegOutputs {  // the kernel parameters it uses, passed by value
    uint16_t *out;
    float *part_o, *part_ml;
    int T, Hq, G;
};

struct SegEndRet {
    uint32_t pair_uses;
    int *ready_ctr;
    bool staged;
    bool ok;
};

template <int MROWS>
__device__ __noinline__ SegEndRet softmax_segment_end(
    const SegOutputs p, TcSmem *sh, const int *tile_base, const PairLane pl, const Cursor cur,
    const long long jt, const long long U, const int nctas, const int nlane, const int myslot,
    const uint32_t tl, const int quarter, const int half, const int hc, const int lane,
    const int warp, const int r, const int rglob, const int kvh, const bool lane_has_row,
    const bool row_valid, const bool warp_active, const bool whole, const bool seg_is_first,
    const bool cl, const float m, const float l, const int arrived, int *ctr, uint32_t pair_uses,
    bool staged) {
    int *ready_ctr = nullptr;
    auto done = [&](bool ok) {
        SegEndRet ret;
        ret.pair_uses = pair_uses;
        ret.ready_ctr = ready_ctr;
        ret.staged = staged;
        ret.ok = ok;
        return ret;
    };
    // The segment's last PV product is waited for only where O is read, so
    // that the row sums' exchange, the merge bookkeeping and a merger's loads
    // of the other partial overlap it (warp-collective: call warp-uniformly).
    auto wait_last_pv = [&]() -> bool {
        if (!warp_wait_bounded(&sh->pv_done[jt % kSBufs], (uint32_t)((jt / kSBufs) & 1)))
            return false;
        tc::fence_after();
        if (warp == 2 && lane == 0) SV_STAMP(11);
        return true;
    };
    // row sum = first half's part + second half's part (same order in both)
    sh->xl[quarter][half][lane] = l;
    if (!group_sync(&sh->pair[quarter], pair_uses)) {
        return done(false);
    }
    const float lrow = sh->xl[quarter][0][lane] + sh->xl[quarter][1][lane];
    if (cl) {
        if (!wait_last_pv()) return done(false);
        // cluster mode: this CTA's share of the group, unnormalised,
        // into the merge buffer (the K/V ring is idle now: every copy
        // has landed and every product has read it)
        cluster_stage<MROWS>(p.part_o + (size_t)blockIdx.x * kClusterSlot<MROWS>,
                             tl + kColO + hc, r, half, lane_has_row, row_valid, m, lrow);
        staged = true;
        if (warp == 2 && lane == 0) SV_STAMP(12);
        tc::fence_before();
        return done(true);
    }
    const int t = row_valid ? rglob / p.G : 0;
    const int g = row_valid ? rglob - t * p.G : 0;
    uint16_t *orow = p.out + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD + hc;
    // A split pair: the last CTA to arrive merges the others'
    // partials into its own O; the others leave a partial and flag it
    // ready once it is visible.  Nobody waits for a CTA that has not
    // already arrived.
    int nc = 1, c0 = 0, slot0 = 0;
    bool merger = whole;
    if (!whole && warp_active) {
        const long long ub = (long long)tile_base[cur.b] * pl.npr + (long long)cur.pi * cur.n;
        c0 = cta_of(U, nctas, ub);  // slots; contributor i is CTA (c0 + i) * nlane + lane
        nc = cta_of(U, nctas, ub + cur.n - 1) - c0 + 1;
        slot0 = cta_begin(U, nctas, c0) >= ub ? 0 : 1;
        const int pos = __shfl_sync(0xffffffffu, arrived, 0);
        merger = pos == nc - 1;
        if (merger) {
            bool ready = true;
            if (lane == 0) {
                const long long t0 = clock64();
                while (ld_acquire_gpu(ctr + kSoftmaxWarps) < nc - 1)
                    if (clock64() - t0 > kWaitCycles) {
                        ready = false;
                        break;
                    }
                if (ready) {
                    ctr[0] = 0;  // ready for the next call
                    ctr[kSoftmaxWarps] = 0;
                }
            }
            if (!__shfl_sync(0xffffffffu, ready, 0)) {
                return done(false);
            }
            __syncwarp();  // the others' partials are read after lane 0's acquire
        }
    }
    if (warp_active) {
        // the other contributors' (max, sum) of this row half
        auto part_slot = [&](int i) -> size_t {
            return (size_t)((c0 + i) * nlane + pl.poff) * 2 + (i == 0 ? slot0 : 0);
        };
        auto part_row = [&](int i) -> size_t { return part_slot(i) * MROWS + r; };
        // O of a partial slot is chunk-major: 16-byte chunk c (columns 4c..4c+3)
        // of row r at float4 (slot * 32 + c) * MROWS + r, so that the lanes of a
        // warp, a row each, store and load consecutive 16 bytes
        auto part_o4 = [&](size_t slot_i, int c) -> size_t {
            return (slot_i * (kD / 4) + (size_t)((hc >> 2) + c)) * MROWS + r;
        };
        // The merge takes the contributors in index order with the same
        // arithmetic whoever merges, so the result does not depend on
        // which CTA finished last.
        const int self = myslot - c0;
        auto ml_of = [&](int i) -> float2 {
            return i == self ? make_float2(m, lrow)
                             : __ldcg(reinterpret_cast<const float2 *>(p.part_ml + part_row(i) * 4 + half * 2));
        };
        float mstar = m, lsum = lrow;
        if (!whole && merger && row_valid && nc != 2) {
            for (int i = 0; i < nc; ++i) mstar = fmaxf(mstar, ml_of(i).x);
            lsum = 0.f;
            for (int i = 0; i < nc; ++i) {
                const float2 ml = ml_of(i);
                const float w = ml.x == kNegInf ? 0.f : ex2_approx(ml.x - mstar);
                lsum = __fmaf_rn(ml.y, w, lsum);
            }
        }
        const int slot = seg_is_first ? 0 : 1;
        float4 *po4 = reinterpret_cast<float4 *>(p.part_o);
        const size_t my_slot = (size_t)blockIdx.x * 2 + slot;
        if (!whole && merger && nc == 2) {  // (the same in every lane)
            // two contributors (the usual split): the other's partial
            // fetched in one go, then the same arithmetic as below
            const int oth = 1 - self;
            const size_t pro = part_row(oth);
            float2 mlo = make_float2(kNegInf, 0.f);
            float4 oo[16];
            const float4 *src = reinterpret_cast<const float4 *>(p.part_o);
            if (row_valid) {
                mlo = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + pro * 4 + half * 2));
    #pragma unroll
                for (int c = 0; c < 16; ++c) oo[c] = __ldcg(src + part_o4(part_slot(oth), c));
            } else {
    #pragma unroll
                for (int c = 0; c < 16; ++c) oo[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (!wait_last_pv()) return done(false);
            const float ms2 = fmaxf(m, mlo.x);
            const float ws = m == kNegInf ? 0.f : ex2_approx(m - ms2);
            const float wo = mlo.x == kNegInf ? 0.f : ex2_approx(mlo.x - ms2);
            const float w0 = self == 0 ? ws : wo, w1 = self == 0 ? wo : ws;
            const float l0 = self == 0 ? lrow : mlo.y, l1 = self == 0 ? mlo.y : lrow;
            const float inv2 = 1.f / __fmaf_rn(l1, w1, __fmaf_rn(l0, w0, 0.f));
    #pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t ov[32];
                __syncwarp();  // converged for the warp-collective load
                tc::tmem_ld32(tl + kColO + hc + 32 * h, ov);
                tc::wait_ld();
                if (!row_valid) continue;
                float acc[32];
    #pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 o = oo[8 * h + c];
                    const float xo[4] = {o.x, o.y, o.z, o.w};
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float xs = __uint_as_float(ov[4 * c + e]);
                        const float x0 = self == 0 ? xs : xo[e], x1 = self == 0 ? xo[e] : xs;
                        acc[4 * c + e] = __fmaf_rn(x1, w1, __fmaf_rn(x0, w0, 0.f));
                    }
                }
    #pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 wv;
                    wv.x = pack_bf16x2(acc[8 * c + 0] * inv2, acc[8 * c + 1] * inv2);
                    wv.y = pack_bf16x2(acc[8 * c + 2] * inv2, acc[8 * c + 3] * inv2);
                    wv.z = pack_bf16x2(acc[8 * c + 4] * inv2, acc[8 * c + 5] * inv2);
                    wv.w = pack_bf16x2(acc[8 * c + 6] * inv2, acc[8 * c + 7] * inv2);
                    *reinterpret_cast<uint4 *>(orow + 32 * h + 8 * c) = wv;
                }
            }
        } else {
        if (!wait_last_pv()) return done(false);
        const float inv = 1.f / lsum;
    #pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t ov[32];
            __syncwarp();  // converged for the warp-collective load
            tc::tmem_ld32(tl + kColO + hc + 32 * h, ov);
            tc::wait_ld();
            if (!row_valid) continue;
            if (merger) {
                float acc[32];
    #pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(ov[j]);
                if (!whole) {
    #pragma unroll
                    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
                    for (int i = 0; i < nc; ++i) {
                        const float2 ml = ml_of(i);
                        const float w = ml.x == kNegInf ? 0.f : ex2_approx(ml.x - mstar);
                        if (i == self) {
    #pragma unroll
                            for (int j = 0; j < 32; ++j) acc[j] = __fmaf_rn(__uint_as_float(ov[j]), w, acc[j]);
                        } else {
                            const float4 *src = reinterpret_cast<const float4 *>(p.part_o);
                            const size_t si = part_slot(i);
    #pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const float4 o = __ldcg(src + part_o4(si, 8 * h + c));
                                acc[4 * c] = __fmaf_rn(o.x, w, acc[4 * c]);
                                acc[4 * c + 1] = __fmaf_rn(o.y, w, acc[4 * c + 1]);
                                acc[4 * c + 2] = __fmaf_rn(o.z, w, acc[4 * c + 2]);
                                acc[4 * c + 3] = __fmaf_rn(o.w, w, acc[4 * c + 3]);
                            }
                        }
                    }
                }
    #pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 wv;
                    wv.x = pack_bf16x2(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
                    wv.y = pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
                    wv.z = pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
                    wv.w = pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
                    *reinterpret_cast<uint4 *>(orow + 32 * h + 8 * c) = wv;
                }
            } else {
    #pragma unroll
                for (int c = 0; c < 8; ++c)
                    po4[part_o4(my_slot, 8 * h + c)] =
                        make_float4(__uint_as_float(ov[4 * c]), __uint_as_float(ov[4 * c + 1]),
                                    __uint_as_float(ov[4 * c + 2]), __uint_as_float(ov[4 * c + 3]));
            }
        }
        }
        if (!merger) {
            if (row_valid)
                *reinterpret_cast<float2 *>(p.part_ml + (((size_t)blockIdx.x * 2 + slot) * MROWS + r) * 4 +
                                            half * 2) = make_float2(m, lrow);
            if (ctr) ready_ctr = ctr + kSoftmaxWarps;  // flagged after the next tile (or at the end)
        }
    }
    if (warp == 2 && lane == 0) SV_STAMP(12);
    tc::fence_before();
    return done(true);
}

// MROWS query rows per group: 128 (M=128 products, row r in TMEM lane r) or
// 64 (M=64 products, row r in lane 32*(r/16) + r%16: lanes 0-15 of each
// 32-lane quarter) for groups of at most 64 rows.
template <int STAGES, int MROWS>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attention_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv,
                             const __grid_constant__ CUtensorMap tmq, const AttnKParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    uint8_t *qbuf = smem + STAGES * kStageBytes;  // 2 x (two 64-dim boxes of MROWS rows)
    constexpr int kQBox = MROWS * 128;            // one 64-dim box: MROWS rows of 128 bytes
    TcSmem *sh = reinterpret_cast<TcSmem *>(qbuf + 2 * 2 * kQBox);
    int *tile_base = reinterpret_cast<int *>(sh + 1);  // [B + 1]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int HR = p.Hkv * p.RG;

    if (tid == 0) SV_STAMP_ENTRY();
    SV_STAMP_EXIT();
    // The set-up that reads no global memory (barriers, tensor-map prefetch,
    // the Q padding rows, the tensor memory) comes before the wait for the
    // previous kernel: with programmatic launch it overlaps that kernel's tail.
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh->full_k[s], 1);
            mbar_init(&sh->empty_k[s], 1);
            mbar_init(&sh->full_v[s], 1);
            mbar_init(&sh->empty_v[s], 1);
        }
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&sh->s_full[i], 1);
            mbar_init(&sh->p_full[i], kSoftmaxWarps);
            mbar_init(&sh->pv_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh->q_full[i], 1);
            mbar_init(&sh->q_empty[i], 1);
        }
        mbar_init(&sh->fin, 1);
        mbar_init(&sh->fin_pv, 1);
        for (int q = 0; q < 4; ++q) mbar_init(&sh->pair[q], 2);
        mbar_init(&sh->k_first, 1);
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmq);
    }
    // Q rows past rows_per_rg (when G does not divide MROWS) are never loaded:
    // zero them once so that the padding rows of S stay finite.
    for (int i = tid; i < 2 * 2 * (MROWS - p.rows_per_rg) * 8; i += kTcThreads) {
        const int per_box = (MROWS - p.rows_per_rg) * 8;  // 16-byte words past the loaded rows
        const int box = i / per_box, w = i - box * per_box;
        *reinterpret_cast<uint4 *>(qbuf + box * kQBox + p.rows_per_rg * 128 + w * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    // no exchange word carries a tag yet (tags start at 1)
    for (int i = tid; i < 2 * 4 * 2 * 32; i += kTcThreads) (&sh->xmax[0][0][0][0])[i] = 0ull;
    tc::fence_proxy_async_smem();
    if (warp == 1) tc::tmem_alloc(&sh->tmem, kTcCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = sh->tmem;

    griddep_wait();
    griddep_launch_dependents();
    if (tid == 0) SV_STAMP(2);
    const int pre_L = tid < p.B ? p.prefix_lens[tid] : 0;
    const int pre_T = tid < p.B ? nodes_of(p, tid) : 0;
    attn_prologue(p, tile_base, kTcThreads, pre_L, pre_T);

    // With several row groups per KV head, the CTAs go in lanes, one per row
    // group: CTA c works in lane c % RG, and the lanes split the (sequence,
    // KV head, tile) units identically, so the RG CTAs of a slot stream the
    // same K/V tiles side by side and all but the first read them from L2.
    //
    // In cluster mode the units of one (sequence, KV head, row group) go to
    // one cluster, CTA k taking the k-th contiguous share of its tiles; no CTA
    // leaves early (all of them meet at the cluster barriers at the end).
    const bool cl = p.cluster > 1;
    const int cs = cl ? p.cluster : 1;
    const int crank = cl ? (int)cluster_ctarank() : 0;
    const int cpair = (int)blockIdx.x / cs;              // cluster mode: the cluster's group
    const int cb = cl ? cpair / HR : 0;                  // its sequence
    const int cpr = cl ? cpair - cb * HR : 0;            // its (KV head, row group)
    const int cn = cl && cb < p.B ? tile_base[cb + 1] - tile_base[cb] : 0;  // its tiles
    const int nlane = cl ? 1 : p.RG;
    const PairLane pl{cl ? HR : nlane > 1 ? p.Hkv : HR, nlane, cl ? 0 : (int)blockIdx.x % nlane};
    const long long U = (long long)tile_base[p.B] * pl.npr;  // units of one lane
    // At least kMinTilesPerCta tiles a slot: below that a CTA's fixed costs
    // (pipeline fill, epilogue) and many-way merges outweigh the parallelism.
    const int slots_max = (int)gridDim.x / nlane;
    const long long want = U / kMinTilesPerCta > 0 ? U / kMinTilesPerCta : 1;
    const int nctas = (int)(want < (long long)slots_max ? want : (long long)slots_max);  // slots in use
    const int myslot = (int)blockIdx.x / nlane;
    if (!cl && myslot >= nctas) {  // no work: give the tensor memory back
        if (warp == 1) tc::tmem_dealloc(tbase, kTcCols);
        return;
    }
    long long u_begin, u_end;
    if (cl) {
        const long long u0 = (long long)tile_base[cb < p.B ? cb : p.B] * HR + (long long)cpr * cn;
        u_begin = u0 + (long long)cn * crank / cs;
        u_end = u0 + (long long)cn * (crank + 1) / cs;
    } else {
        u_begin = cta_begin(U, nctas, myslot);
        u_end = cta_begin(U, nctas, myslot + 1);
    }
    volatile int *abort_flag = &sh->abort_flag;
    if (tid == 0) SV_STAMP(3);

    auto fail = [&](int b) {
        *abort_flag = 1;
        if (p.seq_status) p.seq_status[b] = SV_ERR_TIMEOUT;
    };

    if (warp == 0 || warp == kVLoadWarp) {
        // ================= producers: warp 0 fills the K halves of the ring,
        // the last warp the V halves.  A K half is refilled as soon as the S
        // product that read it is done, a V half once its PV product is, so
        // the next K tiles stream in while a tile's softmax and PV run.
        if (!(p.block_table && p.page_size < kBK)) {
            if (lane == 0) {
                const bool is_k = warp == 0;
                uint64_t *full = is_k ? sh->full_k : sh->full_v;
                uint64_t *empty = is_k ? sh->empty_k : sh->empty_v;
                const CUtensorMap *map = is_k ? &tmk : &tmv;
                const int half_off = is_k ? 0 : 2 * kBox;
                // K/V tiles are streamed: evict-first keeps the stream from
                // pushing code, Q and partials out of L2.  (Among evict-first
                // lines the oldest go first, so a tile still outlives the few
                // microseconds between the reads of the lanes of one slot.)
                const uint64_t pol = l2_policy_evict_first();
                auto load = [&](void *dst, int x, int y, uint64_t *bar) {
                    tma_load_2d_hint(dst, map, x, y, bar, pol);
                };
                Cursor cur = cursor_at(tile_base, p.B, pl, u_begin);
                long long k = 0;
                uint32_t qseg = 0;  // segments whose Q was issued
                if (is_k) SV_STAMP(4);
                for (long long u = u_begin; u < u_end; ++u, ++k) {
                    const int s = (int)(k % STAGES);
                    const uint32_t ph = (uint32_t)((k / STAGES) & 1);
                    // At the start every SM asks for its ring at once: the first V
                    // tile waits until the first K tile (which the first S
                    // product needs) has been requested.
                    if (!is_k && k == 0 && !mbar_wait_bounded(&sh->k_first, 0)) {
                        fail(cur.b);
                        break;
                    }
                    const int kvh = cur.pr / p.RG;
                    const int kb = cur.tile * kBK;
                    if (!p.block_table) {
                        // contiguous caches: the tile is 128 consecutive rows
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                            fail(cur.b);
                            break;
                        }
                        if (*abort_flag) break;
                        const int y = (cur.b * p.Hkv + kvh) * p.S_max + kb;
                        uint8_t *st = smem + s * kStageBytes + half_off;
                        mbar_arrive_expect_tx(&full[s], 2 * kBox);
                        load(st, 0, y, &full[s]);
                        load(st + kBox, 64, y, &full[s]);
                    } else {
                        // paged, pages of 128 slots or more: the tile sits in one page
                        // (its id read before the wait, so the load overlaps it); an
                        // id out of range (reported by the prologue) reads zeros
                        const int pg = p.block_table[(size_t)cur.b * p.max_pages + kb / p.page_size];
                        const int y = (pg >= 0 && pg < p.num_pages)
                                          ? (pg * p.Hkv + kvh) * p.page_size + kb % p.page_size
                                          : -kBK;
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                            fail(cur.b);
                            break;
                        }
                        if (*abort_flag) break;
                        uint8_t *st = smem + s * kStageBytes + half_off;
                        mbar_arrive_expect_tx(&full[s], 2 * kBox);
                        load(st, 0, y, &full[s]);
                        load(st + kBox, 64, y, &full[s]);
                    }
                    if (is_k && k == 0) {
                        mbar_arrive(&sh->k_first);
                        SV_STAMP(6);
                    }
                    if (is_k && (u == u_begin || cur.tile == 0)) {
                        // this segment's Q rows (rows_per_rg of them: rows_per_rg / G
                        // nodes x G heads, a 3-D box) into Q buffer qseg & 1, once
                        // the S products of the segment two back are done; requested
                        // after the segment's first K tile, which comes from HBM while Q
                        // mostly comes from L2
                        const int qb = (int)(qseg & 1);
                        if (!mbar_wait_bounded(&sh->q_empty[qb], ((qseg >> 1) & 1) ^ 1u)) {
                            fail(cur.b);
                            break;
                        }
                        const int kvh = cur.pr / p.RG, rg = cur.pr - kvh * p.RG;
                        const int tpr = p.rows_per_rg / p.G;  // nodes per row group
                        const int z = cur.b * p.T + rg * tpr;
                        uint8_t *qd = qbuf + qb * 2 * kQBox;
                        mbar_arrive_expect_tx(&sh->q_full[qb], 2u * 128u * (uint32_t)p.rows_per_rg);
                        tma_load_3d(qd, &tmq, 0, kvh * p.G, z, &sh->q_full[qb]);
                        tma_load_3d(qd + kQBox, &tmq, 64, kvh * p.G, z, &sh->q_full[qb]);
                        if (qseg == 0) SV_STAMP(5);
                        ++qseg;
                    }
                    if (!is_k && k == 0) SV_STAMP(18);
                    if (is_k) SV_STAMP(10);
                    cursor_next(cur, tile_base, p.B, pl);
                }
                if (is_k && k == 0) mbar_arrive(&sh->k_first);  // none issued: release the V side
                // every copy issued must land before the CTA may exit
                const long long first = k > STAGES ? k - STAGES : 0;
                for (long long j = first; j < k; ++j)
                    mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1));
                for (uint32_t g2 = qseg > 2 ? qseg - 2 : 0; g2 < qseg; ++g2)
                    mbar_wait_bounded(&sh->q_full[g2 & 1], (g2 >> 1) & 1);
            }
        } else {
            // Paged, pages of 8-64 slots: a tile is 128 / page_size blocks of
            // page_size rows, one per page.  Lane i reads page i's id and
            // issues that block's two boxes, so a tile's blocks go out
            // together instead of one after another from one thread.  The
            // waits are the warp's (one verdict for all lanes); lane 0 does
            // the barrier accounting and the Q loads.  (Pages past the
            // sequence's end may hold any id: one out of range reads zeros,
            // and those keys are masked anyway.)
            const bool is_k = warp == 0;
            uint64_t *full = is_k ? sh->full_k : sh->full_v;
            uint64_t *empty = is_k ? sh->empty_k : sh->empty_v;
            const CUtensorMap *map = is_k ? &tmk : &tmv;
            const int half_off = is_k ? 0 : 2 * kBox;
            const uint64_t pol = l2_policy_evict_first();
            const int ps = p.page_size;
            Cursor cur = cursor_at(tile_base, p.B, pl, u_begin);
            long long k = 0;
            uint32_t qseg = 0;
            for (long long u = u_begin; u < u_end; ++u, ++k) {
                const int s = (int)(k % STAGES);
                const uint32_t ph = (uint32_t)((k / STAGES) & 1);
                if (!is_k && k == 0 && !warp_wait_bounded(&sh->k_first, 0)) {
                    fail(cur.b);
                    break;
                }
                if (is_k && (u == u_begin || cur.tile == 0)) {
                    const int qb = (int)(qseg & 1);
                    if (!warp_wait_bounded(&sh->q_empty[qb], ((qseg >> 1) & 1) ^ 1u)) {
                        fail(cur.b);
                        break;
                    }
                    if (lane == 0) {
                        const int kvh = cur.pr / p.RG, rg = cur.pr - kvh * p.RG;
                        const int z = cur.b * p.T + rg * (p.rows_per_rg / p.G);
                        uint8_t *qd = qbuf + qb * 2 * kQBox;
                        mbar_arrive_expect_tx(&sh->q_full[qb], 2u * 128u * (uint32_t)p.rows_per_rg);
                        tma_load_3d(qd, &tmq, 0, kvh * p.G, z, &sh->q_full[qb]);
                        tma_load_3d(qd + kQBox, &tmq, 64, kvh * p.G, z, &sh->q_full[qb]);
                    }
                    ++qseg;
                }
                const int kvh = cur.pr / p.RG;
                const int kb = cur.tile * kBK;
                const int nsub = min(kBK / ps, p.max_pages - kb / ps);
                int y = -kBK;
                if (lane < nsub) {
                    const int pg = p.block_table[(size_t)cur.b * p.max_pages + kb / ps + lane];
                    y = (pg >= 0 && pg < p.num_pages) ? (pg * p.Hkv + kvh) * ps : -kBK;
                }
                if (!warp_wait_bounded(&empty[s], ph ^ 1u)) {
                    fail(cur.b);
                    break;
                }
                if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
                uint8_t *st = smem + s * kStageBytes + half_off;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], 2u * 128u * (uint32_t)(nsub * ps));
                __syncwarp();  // the expected bytes are set before any block lands
                if (lane < nsub) {
                    tma_load_2d_hint(st + lane * ps * 128, map, 0, y, &full[s], pol);
                    tma_load_2d_hint(st + kBox + lane * ps * 128, map, 64, y, &full[s], pol);
                }
                if (is_k && k == 0 && lane == 0) mbar_arrive(&sh->k_first);
                cursor_next(cur, tile_base, p.B, pl);
            }
            if (is_k && k == 0 && lane == 0) mbar_arrive(&sh->k_first);  // none issued
            if (lane == 0) {  // every copy issued must land before the CTA may exit
                const long long first = k > STAGES ? k - STAGES : 0;
                for (long long j = first; j < k; ++j)
                    mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1));
                for (uint32_t g2 = qseg > 2 ? qseg - 2 : 0; g2 < qseg; ++g2)
                    mbar_wait_bounded(&sh->q_full[g2 & 1], (g2 >> 1) & 1);
            }
        }
    } else if (warp == 1 || warp == kPvWarp) {
        // ================= MMA issue: lane 0 of warp 1 the S = Q K^T
        // products, lane 0 of the last warp the O += P V products, each in
        // tile order behind (bounded) blocking waits, so neither polls nor
        // holds back the other (tcgen05.commit tracks its own thread's MMAs).
        if (lane == 0) {
            bool ok = true;
            Cursor cur = cursor_at(tile_base, p.B, pl, u_begin);
            const long long nt = u_end - u_begin;
            if (warp == 1) {
                constexpr uint32_t idS = tc::idesc_bf16(MROWS, kBK, false);
                uint32_t seg = 0;  // segments started
                int sb = 0;        // S buffer of tile j, and the parity of its use
                uint32_t sph = 0;
                for (long long j = 0; j < nt; ++j) {
                    const int s = (int)(j % STAGES);
                    // this segment's Q has landed, the K tile has landed, the S
                    // buffer is free (PV of tile j - kSBufs, whose P lived there, is done)
                    if (j == 0 || cur.tile == 0) {
                        ok = mbar_wait_bounded(&sh->q_full[seg & 1], (seg >> 1) & 1);
                        ++seg;
                    }
                    if (ok) ok = mbar_wait_bounded(&sh->full_k[s], (uint32_t)((j / STAGES) & 1));
                    if (j == 0) SV_STAMP(7);
                    if (ok && j >= kSBufs) ok = mbar_wait_bounded(&sh->pv_done[sb], sph ^ 1u);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    // dims 16kk..: 32 bytes on within a 64-dim box, the next box on
                    const uint64_t dk = tc::smem_desc(base_u32 + s * kStageBytes, 16, 1024);
                    const uint64_t dq = tc::smem_desc(base_u32 + STAGES * kStageBytes +
                                                          (uint32_t)(((seg - 1) & 1) * 2 * kQBox),
                                                      16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint64_t bd = dk + (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2);
                        const uint64_t ad = dq + (uint64_t)((kk >> 2) * (kQBox >> 4) + (kk & 3) * 2);
                        tc::mma_bf16(tbase + kColS + (uint32_t)sb * kBK, ad, bd, idS,
                                     kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&sh->s_full[sb]);
                    if (++sb == kSBufs) {
                        sb = 0;
                        sph ^= 1u;
                    }
                    if (cur.tile == cur.n - 1 || j == nt - 1)
                        tc::commit(&sh->q_empty[(seg - 1) & 1]);  // Q buffer free once these S are done
                    tc::commit(&sh->empty_k[s]);  // the K half may be refilled once S(j) is done
                    cursor_next(cur, tile_base, p.B, pl);
                }
            } else {
                constexpr uint32_t idPV = tc::idesc_bf16(MROWS, kD, true);
                int sb = 0;  // S buffer (holding P) of tile j, and the parity of its use
                uint32_t sph = 0;
                for (long long j = 0; j < nt; ++j) {
                    const int s = (int)(j % STAGES);
                    const bool first = (j == 0) || cur.tile == 0;  // O starts over
                    ok = mbar_wait_bounded(&sh->p_full[sb], sph);
                    if (ok) ok = mbar_wait_bounded(&sh->full_v[s], (uint32_t)((j / STAGES) & 1));
                    if (j == 0) SV_STAMP(19);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    // V rows 16kk.. start 2048 bytes apart (descriptor address units of 16 bytes)
                    const uint64_t dv = tc::smem_desc(base_u32 + s * kStageBytes + 2 * kBox, kBox, 1024);
                    const uint32_t pcol = tbase + kColS + (uint32_t)sb * kBK;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t bd = dv + (uint64_t)(kk * (2048 >> 4));
                        // P of keys 16kk.. : columns 8kk.. of the first half, 64+.. of the second
                        tc::mma_bf16_ts(tbase + kColO, pcol + kk * 8 + (kk >= 4 ? 32 : 0), bd, idPV,
                                        (kk > 0 || !first) ? 1u : 0u);
                    }
                    tc::commit(&sh->pv_done[sb]);
                    if (++sb == kSBufs) {
                        sb = 0;
                        sph ^= 1u;
                    }
                    tc::commit(&sh->empty_v[s]);  // the V half may be refilled once PV(j) is done
                    cursor_next(cur, tile_base, p.B, pl);
                }
            }
            if (!ok) fail(cur.b < p.B ? cur.b : 0);
            // all MMAs this thread issued complete before the TMEM is released
            uint64_t *fin = warp == 1 ? &sh->fin : &sh->fin_pv;
            tc::commit(fin);
            mbar_wait_bounded(fin, 0);
        }
        __syncwarp();
        tc::fence_before();
        named_bar_sync(1, (2 + kSoftmaxWarps) * 32);
        if (warp == 1) {
            tc::fence_after();
            tc::tmem_dealloc(tbase, kTcCols);
        }
    } else {
    // ===================== softmax warps 2..9: two threads per query row
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;      // 0: keys / output columns 0-63, 1: 64-127
    const int hc = 64 * half;
    constexpr int kRowsPerQuarter = MROWS / 4;  // 32, or 16 with M=64
    const bool lane_has_row = lane < kRowsPerQuarter;
    const int r = quarter * kRowsPerQuarter + (lane_has_row ? lane : 0);  // row in the group
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);         // this warp's lanes
    const float sc = p.scale_log2;
    const float2 sc2 = make_float2(sc, sc);
    float m = kNegInf, l = 0.f;
    uint64_t anc = 0;
    uint32_t pair_uses = 0;
    int *ready_ctr = nullptr;  // a partial of this warp waiting to be flagged ready
    bool staged = false;       // cluster mode: this warp's rows are in the merge buffer
    // The warp's partial writes are visible before the ready count moves.
    auto flag_ready = [&](int *c) {
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(c, 1);
        }
        __syncwarp();
    };
    int L = 0, kv_end = 0, seg_first_tile = 0, kvh = 0, rg = 0, rglob = 0;
    bool seg_is_first = true, warp_active = false, row_valid = false;
    int next_L = 0, next_T = 0;  // the next segment's prefix length and nodes, read ahead
    int2 next_par = make_int2(-1, -1);  // and its parents (two nodes a lane)
    bool have_next_L = false;
    const SegOutputs seg_out{p.out, p.part_o, p.part_ml, p.T, p.Hq, p.G};
    Cursor cur = cursor_at(tile_base, p.B, pl, u_begin);
    long long jt = 0, u = u_begin;
    int sb = 0;         // S buffer of tile jt
    uint32_t sph = 0;   // and the parity of its use
    // One tile: the tile at cur, unit u, tile jt of the run; false when a
    // bounded wait gave up.  FULL adds the pieces only some tiles need: a
    // segment's first tile (O starts over; a partial left by the previous
    // segment is flagged ready), the tiles with keys at or past L (the ancestor
    // mask), the segment's last tile in the run (the split pair's counter, the
    // V rows past the sequence's end, the end of the segment).  The tiles in
    // between run the short form, whose code has almost no branches: a taken
    // branch in this loop costs instruction fetch on every tile.
    auto tile = [&](auto full_tag) -> bool {
        constexpr bool FULL = decltype(full_tag)::value;
        const bool first_tile = FULL && cur.tile == seg_first_tile;  // O is overwritten by this tile's PV
        const int kbase = cur.tile * kBK;
        const bool last_of_pair = FULL && cur.tile == cur.n - 1;
        const bool seg_end = FULL && (last_of_pair || u == u_end - 1);
        const bool whole = seg_first_tile == 0 && last_of_pair;
        // The last tile of a split segment: arrive on the pair's counter now
        // (per warp: its rows, its half of the columns), so the atomic's round
        // trip overlaps this tile; the last CTA to arrive merges.
        int *ctr = nullptr;
        int arrived = 0;
        if (FULL && !cl && seg_end && !whole && warp_active) {
            ctr = p.pair_ctr + ((size_t)((cur.b * p.Hkv + kvh) * p.RG + rg) * 2) * kSoftmaxWarps + (warp - 2);
            if (lane == 0) arrived = atomicAdd(ctr, 1);
        }
        const uint32_t sbuf = tl + kColS + (uint32_t)sb * kBK + hc;  // this half's S columns

        // ---- half S row from TMEM; P written back over its first 32 columns
        if (!warp_wait_bounded(&sh->s_full[sb], sph)) return false;
        tc::fence_after();
        if (warp == 2 && lane == 0) {
            if (jt == 0) SV_STAMP(8);
            SV_STAMP(9);
            SV_STAMP_VALUE(17, jt + 1);
        }
        if (warp_active) {
            float sv[64];
            {
                uint32_t ra[32], rb[32];
                tc::tmem_ld32(sbuf, ra);
                tc::tmem_ld32(sbuf + 32, rb);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    sv[j] = __uint_as_float(ra[j]);
                    sv[32 + j] = __uint_as_float(rb[j]);
                }
            }
            const int k0 = kbase + hc;  // key of sv[0]
            if (FULL && k0 + 64 > L) {
                // bit j: key k0 + j visible to this row (a prefix key, or a
                // new node on the row's root path; anc has no bit past T)
                const int dl = L - k0;  // keys before L in this half tile (may be <= 0)
                const uint64_t pre = dl <= 0 ? 0ull : ((1ull << dl) - 1ull);
                const uint64_t nodes = dl >= 0 ? (dl >= 64 ? 0ull : anc << dl)
                                               : (-dl >= 64 ? 0ull : anc >> -dl);
                const uint64_t vis = pre | nodes;
                const uint32_t vlo = (uint32_t)vis, vhi = (uint32_t)(vis >> 32);
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const uint32_t w = j < 32 ? vlo : vhi;
                    if (!((w >> (j & 31)) & 1u)) sv[j] = kNegInf;
                }
            }
            float mq[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
            for (int j = 0; j < 64; ++j) mq[j & 3] = fmaxf(mq[j & 3], sv[j]);
            float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            // the partner holds the other 64 keys of the same rows
            const uint32_t xtag = (uint32_t)jt + 1u;
            xchg_put(&sh->xmax[jt & 1][quarter][half][lane], mx, xtag);
            float mx_other;
            bool ok = xchg_get(&sh->xmax[jt & 1][quarter][half ^ 1][lane], xtag, mx_other);
            mx = fmaxf(mx, mx_other);
            const float c = mx * sc;
            const bool up = c > m + kRescaleThreshold;
            const bool any_up = __any_sync(0xffffffffu, up);
            const float a = up ? ex2_approx(m - c) : 1.f;
            if (up) {
                m = c;
                l *= a;
            }
            const float nb = m == kNegInf ? 0.f : -m;
            const float2 nb2 = make_float2(nb, nb);
            float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float2 tt = __ffma2_rn(make_float2(sv[2 * j], sv[2 * j + 1]), sc2, nb2);
                const float2 e = make_float2(ex2_approx(tt.x), ex2_approx(tt.y));
                if (j & 1) ls1 = __fadd2_rn(ls1, e);
                else ls0 = __fadd2_rn(ls0, e);
                pk[j] = pack_bf16x2(e.x, e.y);
            }
            tc::tmem_st32(sbuf, pk);
            l += (ls0.x + ls0.y) + (ls1.x + ls1.y);
            if (ok && any_up && !first_tile) {
                // O holds earlier tiles of this segment at the old max: once
                // the last PV is done, rescale this half of the row in TMEM
                // (before P is released, so this tile's PV sees it)
                // (tile jt - 1: the buffer before this one)
                ok = rescale_o_half(&sh->pv_done[sb == 0 ? kSBufs - 1 : sb - 1], sb == 0 ? sph ^ 1u : sph,
                                    tl + kColO + hc, a);
            }
            tc::wait_st();
            if (!ok) return false;
        }
        if (FULL && last_of_pair && kbase + kBK > kv_end) {
            // V rows past the sequence's last slot may hold anything (even NaN,
            // and 0 * NaN is NaN in the product): zero them in this stage,
            // once its V half has landed.  With more S buffers than stages the
            // softmax can run ahead of the PV product that last read this
            // stage (tile jt - STAGES), and the stage's barrier could then
            // still show that tile's phase: that product is waited for first.
            if (jt >= STAGES) {
                const long long jo = jt - STAGES;
                if (!warp_wait_bounded(&sh->pv_done[jo % kSBufs], (uint32_t)((jo / kSBufs) & 1)))
                    return false;
            }
            if (!zero_v_tail(&sh->full_v[jt % STAGES], (uint32_t)((jt / STAGES) & 1),
                             smem + (int)(jt % STAGES) * kStageBytes + 2 * kBox, kv_end - kbase,
                             (warp - 2) * 32 + lane))
                return false;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[sb]);
        if (FULL && ready_ctr) {  // the partial left at the previous tile has drained by now
            flag_ready(ready_ctr);
            ready_ctr = nullptr;
        }

        // ---- end of a segment: this half of the O row out of TMEM
        if (FULL && seg_end) {
            const SegEndRet se = softmax_segment_end<MROWS>(
                seg_out, sh, tile_base, pl, cur, jt, U, nctas, nlane, myslot, tl, quarter, half, hc, lane,
                warp, r, rglob, kvh, lane_has_row, row_valid, warp_active, whole, seg_is_first, cl, m,
                l, arrived, ctr, pair_uses, staged);
            pair_uses = se.pair_uses;
            ready_ctr = se.ready_ctr;
            staged = se.staged;
            if (!se.ok) return false;
        }
        cursor_next(cur, tile_base, p.B, pl);
        ++u;
        ++jt;
        if (++sb == kSBufs) {  // (sb, sph) = (jt % kSBufs, (jt / kSBufs) & 1)
            sb = 0;
            sph ^= 1u;
        }
        return true;
    };
    while (u < u_end) {
        // ---- a segment: the tiles of one (sequence, KV head, row group) in this run
        kvh = cur.pr / p.RG;
        rg = cur.pr - kvh * p.RG;
        L = have_next_L ? next_L : p.prefix_lens[cur.b];
        const int Tb = have_next_L ? next_T : nodes_of(p, cur.b);
        const int2 par = have_next_L ? next_par : load_parents_warp(p.parents, p.T, cur.b, lane);
        have_next_L = false;
        kv_end = L + Tb;
        seg_first_tile = cur.tile;
        seg_is_first = (u == u_begin);
        // the group's rows are rows_per_rg (a multiple of G) of the MMA's
        // MROWS; the others are padding
        rglob = rg * p.rows_per_rg + r;
        row_valid = lane_has_row && r < p.rows_per_rg && rglob < p.M && rglob / p.G < Tb;
        warp_active = quarter * kRowsPerQuarter < p.rows_per_rg &&
                      rg * p.rows_per_rg + quarter * kRowsPerQuarter < p.M;
        m = kNegInf;
        l = 0.f;
        anc = ancestors_warp(p.parents == nullptr, par.x, par.y, rglob / p.G, row_valid);
        // tiles of the segment in this run (t0 ..); the first this warp masks
        // (its keys reach L); the tiles after the first and before those run
        // the short form
        int left = (int)min((long long)(cur.n - cur.tile), u_end - u);
        const int t0 = cur.tile;
        const int lm = L - hc - 64;
        const int t_short_end = min(lm < 0 ? 0 : lm / kBK + 1, t0 + left - 1);
        bool ok = true, shorts_done = false;
        while (ok && left > 0) {
            ok = tile(std::true_type{});
            --left;
            if (ok && left > 0 && !shorts_done) {
                shorts_done = true;
                const int t_early = max(t0 + 1, t_short_end - 4);
                while (ok && cur.tile < t_early) {
                    ok = tile(std::false_type{});
                    --left;
                }
                if (ok && u + (cur.n - cur.tile) < u_end) {
                    // the next segment's prefix length, node count and parents, read
                    // a few tiles before this one ends (its Q is brought in by the producer)
                    Cursor nx = cur;
                    nx.tile = nx.n - 1;
                    cursor_next(nx, tile_base, p.B, pl);
                    next_L = p.prefix_lens[nx.b];
                    next_T = nodes_of(p, nx.b);
                    next_par = load_parents_warp(p.parents, p.T, nx.b, lane);
                    have_next_L = true;
                }
                while (ok && cur.tile < t_short_end) {
                    ok = tile(std::false_type{});
                    --left;
                }
            }
        }
        if (!ok) {
            fail(cur.b);
            break;
        }
    }
    if (ready_ctr) flag_ready(ready_ctr);
    if (cl && !staged && lane_has_row && half == 0) {
        // no tile of the group fell to this CTA (or a wait gave up): an empty share
        __stcg(reinterpret_cast<float2 *>(p.part_o + (size_t)blockIdx.x * kClusterSlot<MROWS> +
                                          MROWS * kD) + r,
               make_float2(kNegInf, 0.f));
    }
    tc::fence_before();
    named_bar_sync(1, (2 + kSoftmaxWarps) * 32);
    }  // softmax warps

    if (p.cluster > 1) {
        // (the cluster's group again, rather than kept live through the loop)
        const int cs = p.cluster;
        const int crank = (int)cluster_ctarank();
        const int cb = (int)blockIdx.x / cs / HR, cpr = (int)blockIdx.x / cs - cb * HR;
        const int cn = cb < p.B ? tile_base[cb + 1] - tile_base[cb] : 0;
        // Every CTA's share is in the workspace once all have passed the
        // barrier; then each finishes its own rows.
        cluster_sync_any();
        if (tid == 64) SV_STAMP(13);
        if (p.hook.step_ctr && crank == 0 && !(warp >= 2 && warp < 2 + kSoftmaxWarps)) {
            // fused tree step: every CTA of the cluster has read its tiles, so
            // this row group is done with (sequence cb, KV head kvh); the last
            // of its row groups and the walk to arrive moves the path's rows
            const int kvh = cpr / p.RG;
            // warps 0-1 -> 0..63, warps 2 + kSoftmaxWarps .. (10, 11) -> 64..127
            const int t128 = warp < 2 ? tid : tid - 32 * kSoftmaxWarps;
            int *ctr = p.hook.step_ctr + (size_t)cb * p.Hkv + kvh;
            if (t128 == 0) {
                const int old = atomicAdd(ctr, 1);
                sh->hook_last = old == p.hook.rg_count;
            }
            __syncwarp();
            named_bar_sync(2, 128);
            if (sh->hook_last) {
                __threadfence();  // the walk's path, written before its arrival
                hook_move_rows(p, cb, kvh, reinterpret_cast<uint4 *>(smem), t128, 2);
                if (t128 == 0) *ctr = 0;  // ready for the next call
            }
        }
        if (warp >= 2 && warp < 2 + kSoftmaxWarps) {
            const int kvh = cpr / p.RG, rg = cpr - kvh * p.RG;
            const size_t c0 = (size_t)(blockIdx.x - crank);  // the cluster's first CTA
            const float *slot0 = p.part_o + c0 * kClusterSlot<MROWS>;
            cluster_merge<MROWS>(p, slot0, kClusterSlot<MROWS>, cs, crank, cb, kvh, rg, cn, tid - 64);
#ifdef SV_PHASE_STAMPS
            if (tid == 64) SV_STAMP(20);
            cluster_merge<MROWS>(p, slot0, kClusterSlot<MROWS>, cs, crank, cb, kvh, rg, cn, tid - 64);
            if (tid == 64) SV_STAMP(21);
#endif
        }
        if (tid == 64) SV_STAMP(15);
    }
    if (tid == 0) SV_STAMP(16);
}

// ---------------------------------------------------------------- host side

int tc_smem_bytes(int stages, int mrows, int B) {
    return 1024 + stages * kStageBytes + 2 * 2 * mrows * 128 + (int)sizeof(TcSmem) + (B + 1) * 4;
}

#ifdef SV_PHASE_STAMPS
}  // namespace sv
// Copies the phase stamps of the last attention launch (kStampSlots per CTA,
// CTA-major) to host memory; diagnostic builds only.
extern "C" int sv_debug_attention_stamps(long long *dst, int ctas) {
    if (ctas > sv::kStampCtas) ctas = sv::kStampCtas;
    return cudaMemcpyFromSymbol(dst, sv::g_stamps, sizeof(long long) * ctas * sv::kStampSlots) ==
                   cudaSuccess
               ? 0
               : -1;
}
extern "C" int sv_debug_attention_clear(void) {
    static long long zeros[sv::kStampCtas * sv::kStampSlots];
    return cudaMemcpyToSymbol(sv::g_stamps, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
namespace sv {
#endif

const void *tc_kernel_fn(int stages, int mrows) {
    if (stages == 3 && mrows == 128) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<3, 128>);
    if (stages == 3 && mrows == 64) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<3, 64>);
    if (stages == 2 && mrows == 128) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<2, 128>);
    if (stages == 2 && mrows == 64) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<2, 64>);
    return nullptr;
}

}  // namespace sv
