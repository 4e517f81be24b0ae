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
// the flat list of (sequence, KV head, 128-row group, 64-key tile) units; a
// persistent grid (one CTA per SM) takes equal contiguous ranges of it, so the
// load is balanced whatever the prefix lengths.  A (sequence, KV head) whose
// tiles fall to several CTAs leaves one partial (O, max, sum) per CTA, merged
// afterwards by the combine kernel below.  Inside a CTA (6 warps):
//
//   warp 0      TMA producer: K and V tiles (2-D tensor maps, 128-byte
//               swizzle) into a ring of STAGES shared-memory stages.
//   warp 1      owns the tensor memory (512 columns); one lane issues the
//               MMAs: S = Q K^T (M=128 or 64 rows, N=128 keys, K=128) into
//               one of two TMEM S buffers, and O += P V (N=128, K=128 keys)
//               into the TMEM O accumulator.  Q and P are read from TMEM, K
//               (K-major) and V (MN-major) from the shared-memory ring.  The
//               tiles are 128 keys wide because a product's issue and
//               completion take about the same time for small and large
//               shapes: fewer, larger MMAs keep the tensor pipe fed.
//   warps 2-5   softmax: thread r owns query row r (TMEM lane r).  It reads
//               its S row from TMEM, applies the ancestor mask (a 64-bit set
//               of tree ancestors per row, only in the tile(s) holding the T
//               new rows), keeps the running max (moved only when it grows by
//               more than 2^8, the O row then rescaled in TMEM) and row sum,
//               writes its bf16 P row over the S row it came from in TMEM
//               (the A operand of the PV MMA), and
//               at the end of a segment reads its O row back and writes the
//               output row or its partial.
//
// The MMA lane polls its barriers and issues S of the next tile and PV of the
// oldest pending tile whenever either is ready, so the softmax of one tile
// overlaps the products of its neighbours and no K/V stage is held longer
// than its own tile needs.  Every wait is bounded (SV_ERR_TIMEOUT on expiry);
// the TMEM is always released.
#include "sv_attn_common.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kTcThreads = 192;  // 6 warps
// Tensor-memory columns (32-bit each, one row per lane): two S buffers
// (128 f32 each; the bf16 P row of a tile overwrites the first 64 columns of
// its S row), the O accumulator (128 f32) and the Q tile (128 bf16 = 64
// columns).  Q and P are the A operands of the two products, read by the
// tensor core straight from TMEM, so shared memory holds only the K/V ring.
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;

// Byte offset of 16-byte chunk c (0..7) of row `row` in a 128-byte-swizzled
// block whose rows are 128 bytes (the layout TMA writes with SWIZZLE_128B and
// the tensor core reads with swizzle mode 2).  Used to zero V rows.
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4));
}

struct TcSmem {
    uint64_t full[4], empty[4];  // TMA ring
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t q_full, fin;
    uint32_t tmem;
    int abort_flag;
};

// MROWS query rows per group: 128 (M=128 products, row r in TMEM lane r) or
// 64 (M=64 products, row r in lane 32*(r/16) + r%16: lanes 0-15 of each
// 32-lane quarter) for groups of at most 64 rows.
template <int STAGES, int MROWS>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attention_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const AttnKParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    TcSmem *sh = reinterpret_cast<TcSmem *>(smem + STAGES * kStageBytes);
    int *tile_base = reinterpret_cast<int *>(sh + 1);  // [B + 1]
    int *scan_tmp = tile_base + (p.B + 1);             // [kTcThreads]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int HR = p.Hkv * p.RG;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh->s_full[i], 1);
            mbar_init(&sh->p_full[i], 4);
            mbar_init(&sh->pv_done[i], 1);
        }
        mbar_init(&sh->q_full, 4);
        mbar_init(&sh->fin, 1);
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    attn_prologue(p, tile_base, scan_tmp, kTcThreads);

    const long long U = (long long)tile_base[p.B] * HR;
    const int nctas = (int)(U < (long long)gridDim.x ? U : (long long)gridDim.x);
    if ((int)blockIdx.x >= nctas) return;
    const long long u_begin = cta_begin(U, nctas, blockIdx.x);
    const long long u_end = cta_begin(U, nctas, blockIdx.x + 1);
    volatile int *abort_flag = &sh->abort_flag;

    if (warp == 1) tc::tmem_alloc(&sh->tmem, kTcCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = sh->tmem;

    auto fail = [&](int b) {
        *abort_flag = 1;
        if (p.seq_status) p.seq_status[b] = SV_ERR_TIMEOUT;
    };

    if (warp == 0) {
        // ================= producer
        if (lane == 0) {
            Cursor cur = cursor_at(tile_base, p.B, HR, u_begin);
            long long k = 0;
            for (long long u = u_begin; u < u_end; ++u, ++k) {
                const int s = (int)(k % STAGES);
                const uint32_t ph = (uint32_t)((k / STAGES) & 1);
                if (!mbar_wait_bounded(&sh->empty[s], ph ^ 1u)) {
                    fail(cur.b);
                    break;
                }
                if (*abort_flag) break;
                const int kvh = cur.pr / p.RG;
                const int y = (cur.b * p.Hkv + kvh) * p.S_max + cur.tile * kBK;
                uint8_t *st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&sh->full[s], kStageBytes);
                tma_load_2d(st, &tmk, 0, y, &sh->full[s]);
                tma_load_2d(st + kBox, &tmk, 64, y, &sh->full[s]);
                tma_load_2d(st + 2 * kBox, &tmv, 0, y, &sh->full[s]);
                tma_load_2d(st + 3 * kBox, &tmv, 64, y, &sh->full[s]);
                cursor_next(cur, tile_base, p.B, HR);
            }
            // every copy issued must land before the CTA may exit
            const long long first = k > STAGES ? k - STAGES : 0;
            for (long long j = first; j < k; ++j)
                mbar_wait_bounded(&sh->full[j % STAGES], (uint32_t)((j / STAGES) & 1));
        }
        return;
    }

    if (warp == 1) {
        // ================= MMA issue (one lane)
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(MROWS, kBK, false);
            constexpr uint32_t idPV = tc::idesc_bf16(MROWS, kD, true);
            // Event loop: S of the next tile as soon as its K tile has landed
            // and its TMEM buffer is free (PV of tile j-2, whose P lived
            // there, is done), PV of the oldest pending tile as soon as its P
            // rows are written; never one product waiting on an unrelated one.
            bool ok = true;
            Cursor cur = cursor_at(tile_base, p.B, HR, u_begin);
            const long long nt = u_end - u_begin;
            long long s_next = 0, pv_next = 0;
            uint32_t seg = 0, first_bits = 0;  // bit (j & 31): tile j opens a segment
            bool q_seen = false;
            long long t_progress = clock64();
            while (pv_next < nt) {
                bool progressed = false;
                if (s_next < nt && s_next - pv_next < 2) {
                    const bool new_seg = (s_next == 0) || cur.tile == 0;
                    bool can = !(new_seg && pv_next < s_next);  // finish the old segment first
                    if (can && new_seg && !q_seen) {
                        q_seen = mbar_test_wait(&sh->q_full, seg & 1);
                        can = q_seen;
                    }
                    const int s = (int)(s_next % STAGES);
                    if (can) can = mbar_test_wait(&sh->full[s], (uint32_t)((s_next / STAGES) & 1));
                    if (can && s_next >= 2)
                        can = mbar_test_wait(&sh->pv_done[s_next & 1], (uint32_t)(((s_next - 2) >> 1) & 1));
                    if (can) {
                        tc::fence_after();
                        const uint32_t kbase_sm = base_u32 + s * kStageBytes;
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t bd =
                                tc::smem_desc(kbase_sm + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
                            tc::mma_bf16_ts(tbase + kColS + (uint32_t)(s_next & 1) * kBK,
                                            tbase + kColQ + kk * 8, bd, idS, kk > 0 ? 1u : 0u);
                        }
                        tc::commit(&sh->s_full[s_next & 1]);
                        if (new_seg) {
                            first_bits |= 1u << (s_next & 31);
                            ++seg;
                            q_seen = false;
                        } else {
                            first_bits &= ~(1u << (s_next & 31));
                        }
                        cursor_next(cur, tile_base, p.B, HR);
                        ++s_next;
                        progressed = true;
                    }
                }
                if (pv_next < s_next &&
                    mbar_test_wait(&sh->p_full[pv_next & 1], (uint32_t)((pv_next >> 1) & 1))) {
                    tc::fence_after();
                    const int s = (int)(pv_next % STAGES);
                    const bool first = (first_bits >> (pv_next & 31)) & 1u;
                    const uint32_t vbase = base_u32 + s * kStageBytes + 2 * kBox;
                    const uint32_t pcol = tbase + kColS + (uint32_t)(pv_next & 1) * kBK;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t bd = tc::smem_desc(vbase + kk * 2048, kBox, 1024);
                        tc::mma_bf16_ts(tbase + kColO, pcol + kk * 8, bd, idPV,
                                        (kk > 0 || !first) ? 1u : 0u);
                    }
                    tc::commit(&sh->pv_done[pv_next & 1]);
                    tc::commit(&sh->empty[s]);
                    ++pv_next;
                    progressed = true;
                }
                if (progressed) {
                    t_progress = clock64();
                } else if (clock64() - t_progress > kWaitCycles || *abort_flag) {
                    ok = false;
                    break;
                }
            }
            if (!ok) fail(cur.b < p.B ? cur.b : 0);
            // all MMAs this thread issued complete before the TMEM is released
            tc::commit(&sh->fin);
            mbar_wait_bounded(&sh->fin, 0);
        }
        __syncwarp();
        tc::fence_before();
        named_bar_sync(1, 5 * 32);
        tc::fence_after();
        tc::tmem_dealloc(tbase, kTcCols);
        return;
    }

    // ===================== softmax warps 2..5: one thread per query row
    const int quarter = warp & 3;
    constexpr int kRowsPerQuarter = MROWS / 4;  // 32, or 16 with M=64
    const bool lane_has_row = lane < kRowsPerQuarter;
    const int r = quarter * kRowsPerQuarter + (lane_has_row ? lane : 0);  // row in the group
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);         // this warp's lanes
    const float sc = p.scale_log2;
    float m = kNegInf, l = 0.f;
    uint64_t anc = 0;
    int L = 0, kv_end = 0, seg_first_tile = 0, kvh = 0, rg = 0, rglob = 0;
    bool seg_is_first = true, warp_active = false, row_valid = false;
    Cursor cur = cursor_at(tile_base, p.B, HR, u_begin);
    long long jt = 0;
    for (long long u = u_begin; u < u_end; ++u, ++jt) {
        const bool new_seg = (u == u_begin) || cur.tile == 0;
        if (new_seg) {
            kvh = cur.pr / p.RG;
            rg = cur.pr - kvh * p.RG;
            L = p.prefix_lens[cur.b];
            kv_end = L + p.T;
            seg_first_tile = cur.tile;
            seg_is_first = (u == u_begin);
            rglob = rg * MROWS + r;
            row_valid = lane_has_row && rglob < p.M;
            warp_active = rg * MROWS + quarter * kRowsPerQuarter < p.M;
            m = kNegInf;
            l = 0.f;
            int t = 0, g = 0;
            if (row_valid) {
                t = rglob / p.G;
                g = rglob - t * p.G;
                anc = ancestors(p.parents, p.T, cur.b, t);
            }
            // this thread's Q row into the TMEM A tile (zeros past M); the
            // previous segment's products have all completed (its epilogue
            // waited for its last PV)
            if (warp_active) {
                const uint4 *qsrc = reinterpret_cast<const uint4 *>(
                    p.q + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = row_valid ? qsrc[8 * h + c] : make_uint4(0u, 0u, 0u, 0u);
                        w[4 * c] = v.x;
                        w[4 * c + 1] = v.y;
                        w[4 * c + 2] = v.z;
                        w[4 * c + 3] = v.w;
                    }
                    tc::tmem_st32(tl + kColQ + 32 * h, w);
                }
                tc::wait_st();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->q_full);
            if (cur.tile == 0 && warp == 2 && lane == 0) {
                // this CTA holds the pair's first tile: record who shares the pair
                const long long ub = (long long)tile_base[cur.b] * HR + (long long)cur.pr * cur.n;
                const int c_last = cta_of(U, nctas, ub + cur.n - 1);
                p.pair_info[(cur.b * p.Hkv + kvh) * p.RG + rg] =
                    make_int4((int)blockIdx.x, c_last - (int)blockIdx.x + 1,
                              cta_begin(U, nctas, blockIdx.x) >= ub ? 0 : 1, 0);
            }
        }
        const bool first_tile = new_seg;  // O is overwritten by this tile's PV
        const int kbase = cur.tile * kBK;
        const bool last_of_pair = cur.tile == cur.n - 1;
        const uint32_t sbuf = tl + kColS + (uint32_t)(jt & 1) * kBK;

        // ---- S row from TMEM; P written back over it
        if (!mbar_wait_bounded(&sh->s_full[jt & 1], (uint32_t)((jt >> 1) & 1))) {
            fail(cur.b);
            break;
        }
        tc::fence_after();
        if (warp_active) {
            float sv[kBK];
#pragma unroll
            for (int h = 0; h < kBK / 32; ++h) {
                uint32_t ra[32];
                tc::tmem_ld32(sbuf + 32 * h, ra);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[32 * h + j] = __uint_as_float(ra[j]);
            }
            if (kbase + kBK > L) {
#pragma unroll
                for (int j = 0; j < kBK; ++j) {
                    const int key = kbase + j;
                    const bool allowed =
                        key < L || (key < kv_end && ((anc >> (unsigned)(key - L)) & 1ull));
                    if (!allowed) sv[j] = kNegInf;
                }
            }
            float mx = kNegInf;
#pragma unroll
            for (int j = 0; j < kBK; ++j) mx = fmaxf(mx, sv[j]);
            const float c = mx * sc;
            const bool up = c > m + kRescaleThreshold;
            bool ok = true;
            if (__any_sync(0xffffffffu, up)) {
                const float a = up ? ex2_approx(m - c) : 1.f;
                if (!first_tile) {
                    // O holds earlier tiles of this segment: wait for the last PV, rescale in TMEM
                    ok = mbar_wait_bounded(&sh->pv_done[(jt - 1) & 1], (uint32_t)(((jt - 1) >> 1) & 1));
                    tc::fence_after();
#pragma unroll
                    for (int h = 0; h < kD / 32; ++h) {
                        uint32_t ov[32];
                        tc::tmem_ld32(tl + kColO + 32 * h, ov);
                        tc::wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * a);
                        tc::tmem_st32(tl + kColO + 32 * h, ov);
                    }
                }
                if (up) {
                    m = c;
                    l *= a;
                }
            }
            const float nb = m == kNegInf ? 0.f : -m;
            float ls = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float e0 = ex2_approx(fmaf(sv[64 * h + 2 * j], sc, nb));
                    const float e1 = ex2_approx(fmaf(sv[64 * h + 2 * j + 1], sc, nb));
                    ls += e0 + e1;
                    pk[j] = pack_bf16x2(e0, e1);
                }
                tc::tmem_st32(sbuf + 32 * h, pk);  // P columns 0..63 of this S buffer
            }
            tc::wait_st();
            l += ls;
            if (!ok) {
                fail(cur.b);
                break;
            }
        }
        if (last_of_pair && kbase + kBK > kv_end) {
            // V rows past the sequence's last slot may hold anything (even NaN,
            // and 0 * NaN is NaN in the product): zero them in this stage
            const int z0 = kv_end - kbase;
            uint8_t *vst = smem + (int)(jt % STAGES) * kStageBytes + 2 * kBox;
            for (int i = (quarter * 32 + lane); i < (kBK - z0) * 16; i += 128) {
                const int row = z0 + (i >> 4), c = i & 15;
                *reinterpret_cast<uint4 *>(vst + (c >> 3) * kBox + sw128(row, c & 7)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            tc::fence_proxy_async_smem();
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[jt & 1]);

        // ---- end of a segment: O row out of TMEM
        if (last_of_pair || u == u_end - 1) {
            if (!mbar_wait_bounded(&sh->pv_done[jt & 1], (uint32_t)((jt >> 1) & 1))) {
                fail(cur.b);
                break;
            }
            tc::fence_after();
            const bool whole = seg_first_tile == 0 && last_of_pair;
            const int t = row_valid ? rglob / p.G : 0;
            const int g = row_valid ? rglob - t * p.G : 0;
            uint16_t *orow = p.out + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
            const int slot = seg_is_first ? 0 : 1;
            float *po = p.part_o + (((size_t)blockIdx.x * 2 + slot) * MROWS + r) * kD;
            float *pml = p.part_ml + (((size_t)blockIdx.x * 2 + slot) * MROWS + r) * 2;
            const float inv = 1.f / l;
            if (warp_active) {
#pragma unroll
                for (int h = 0; h < kD / 32; ++h) {
                    uint32_t ov[32];
                    tc::tmem_ld32(tl + kColO + 32 * h, ov);
                    tc::wait_ld();
                    if (!row_valid) continue;
                    if (whole) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv);
                            *reinterpret_cast<uint4 *>(orow + 32 * h + 8 * c) = w;
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<float4 *>(po + 32 * h + 4 * c) =
                                make_float4(__uint_as_float(ov[4 * c]), __uint_as_float(ov[4 * c + 1]),
                                            __uint_as_float(ov[4 * c + 2]), __uint_as_float(ov[4 * c + 3]));
                    }
                }
            }
            tc::fence_before();
            if (!whole && row_valid) *reinterpret_cast<float2 *>(pml) = make_float2(m, l);
        }
        cursor_next(cur, tile_base, p.B, HR);
    }
    tc::fence_before();
    named_bar_sync(1, 5 * 32);
}

// ---------------------------------------------------------------- split merge

// Merge the partials of every (sequence, KV head, row group) whose tiles fell
// to several CTAs: out = sum_c 2^(m_c - m*) O_c / sum_c 2^(m_c - m*) l_c.
// One warp per query row, lanes across the 128 columns; pairs held by one
// CTA (written directly by the attention kernel) and invalid sequences exit.
constexpr int kCombineRows = 8;  // rows (warps) per CTA

__global__ void __launch_bounds__(kCombineRows * 32)
    attention_combine_kernel(const AttnKParams p) {
    const int chunks = p.rows_per_rg / kCombineRows;
    const int pair = blockIdx.x / chunks;
    const int r = (blockIdx.x - pair * chunks) * kCombineRows + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int b = pair / (p.Hkv * p.RG);
    const int rem = pair - b * p.Hkv * p.RG;
    const int kvh = rem / p.RG, rg = rem - kvh * p.RG;
    const int L = p.prefix_lens[b];
    if (L < 0 || (long long)L + p.T > p.S_max) return;
    const int rglob = rg * p.rows_per_rg + r;
    if (rglob >= p.M) return;
    const int4 info = __ldcg(p.pair_info + pair);
    const int nc = info.y;
    if (nc <= 1) return;
    auto row_index = [&](int i) -> size_t {  // contributor i's partial row
        const int slot = i == 0 ? info.z : 0;
        return ((size_t)(info.x + i) * 2 + slot) * p.rows_per_rg + r;
    };
    float mstar = kNegInf;
    for (int i = lane; i < nc; i += 32) mstar = fmaxf(mstar, __ldcg(p.part_ml + row_index(i) * 2));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
    float lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < nc; base += 32) {
        float w = 0.f;
        const int i = base + lane;
        if (i < nc) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + row_index(i) * 2));
            w = ml.x == kNegInf ? 0.f : exp2f(ml.x - mstar);
            lsum += ml.y * w;
        }
        const int cnt = min(32, nc - base);
        for (int j = 0; j < cnt; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_o + row_index(base + j) * kD) + lane);
            acc.x += v.x * wj;
            acc.y += v.y * wj;
            acc.z += v.z * wj;
            acc.w += v.w * wj;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    const float inv = 1.f / lsum;
    const int t = rglob / p.G, g = rglob - t * p.G;
    uint16_t *orow = p.out + (((size_t)b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(orow + lane * 4) = pk;
}

// ---------------------------------------------------------------- host side

int tc_smem_bytes(int stages, int B) {
    return 1024 + stages * kStageBytes + (int)sizeof(TcSmem) + (B + 1) * 4 + kTcThreads * 4;
}

const void *tc_kernel_fn(int stages, int mrows) {
    if (stages == 3 && mrows == 128) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<3, 128>);
    if (stages == 3 && mrows == 64) return reinterpret_cast<const void *>(&tree_attention_tc_kernel<3, 64>);
    return nullptr;
}

sv_status launch_combine(const AttnKParams &p, cudaStream_t st) {
    const unsigned grid = (unsigned)(p.B * p.Hkv * p.RG * (p.rows_per_rg / kCombineRows));
    attention_combine_kernel<<<grid, kCombineRows * 32, 0, st>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv
