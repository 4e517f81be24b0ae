// sv_attention.cu -- verification attention over a prefix KV cache plus each
// node's tree ancestors, with grouped-query heads.
//
// Source: "Chapitre 9 -- Décodage spéculatif" §9.1 (one forward over the
// prefix concatenated with the candidates; the pass stays memory-bound) and
// §9.2 (EAGLE-2 draft tree verified in one attention pass with a custom
// mask); "Parallel Decoding" glossary, Medusa "Tree attention" and
// "L'attention en arbre : la brique commune".
//
// Design (one GPU, HBM-bound by the K/V stream):
//   * The G = Hq/Hkv query heads of a KV head and the T nodes form M = G*T
//     query rows that share every K/V tile, so each tile is read from HBM
//     once per (sequence, KV head) and feeds M rows of tensor-core work.
//   * Work is the flat list of units (sequence b, KV head, row group, 64-key
//     tile).  A persistent grid of CTAs takes equal contiguous ranges of
//     that list, so the load is balanced whatever the prefix lengths; a
//     (sequence, KV head) that straddles CTAs is merged by whichever CTA
//     finishes it last (arrival counter, no waiting between CTAs).
//   * Per CTA: one producer warp issues 2-D TMA copies (128-byte swizzle) of
//     K and V tiles into a multi-stage mbarrier ring; NWC consumer warps own
//     16 query rows each and run QK^T and PV with mma.sync m16n8k16 (bf16 in,
//     f32 accumulate), online softmax in the log2 domain whose running max
//     moves only when it grows by more than 2^8.
//   * The ancestor mask is a 64-bit set per row built by walking the parent
//     array; it only applies to the tile(s) holding the T new rows.
//   * Every wait is bounded; on expiry the CTA records SV_ERR_TIMEOUT for the
//     sequence and winds down after its TMA copies in flight have landed.
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kD = 128;
constexpr int kBK = 64;                   // keys per tile
constexpr int kBox = kBK * 64 * 2;        // one 64-key x 64-dim bf16 TMA box: 8 KB
constexpr int kStageBytes = 4 * kBox;     // K lo/hi + V lo/hi: 32 KB
constexpr int kMaxB = 4096;
constexpr int kMaxT = 64;

struct AttnKParams {
    const uint16_t *q;
    uint16_t *out;
    const int32_t *prefix_lens;
    const int32_t *parents;
    int32_t *seq_status;
    int B, T, Hq, Hkv, G, S_max, M, RG, rows_per_rg;
    float scale_log2;
    float *part_o;   // [grid][2][rows_per_rg][kD]
    float *part_ml;  // [grid][2][rows_per_rg][2]
    int *counters;   // [B][Hkv][RG]
};

// Position in the unit list: sequence, (kv head * RG + row group), tile.
struct Cursor {
    int b, pr, tile, n;
};

__device__ __forceinline__ long long cta_begin(long long U, int grid, int c) {
    return (U * c) / grid;
}

// Index of the CTA whose range holds unit u.
__device__ __forceinline__ int cta_of(long long U, int grid, long long u) {
    return (int)(((u + 1) * grid + U - 1) / U) - 1;
}

__device__ __forceinline__ Cursor cursor_at(const int *tile_base, int B, int HR, long long u) {
    int lo = 0, hi = B - 1;  // last b with tile_base[b] * HR <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)tile_base[mid] * HR <= u) lo = mid;
        else hi = mid - 1;
    }
    Cursor c;
    c.b = lo;
    c.n = tile_base[lo + 1] - tile_base[lo];
    const long long rem = u - (long long)tile_base[lo] * HR;
    c.pr = c.n > 0 ? (int)(rem / c.n) : 0;
    c.tile = c.n > 0 ? (int)(rem - (long long)c.pr * c.n) : 0;
    return c;
}

__device__ __forceinline__ void cursor_next(Cursor &c, const int *tile_base, int B, int HR) {
    if (++c.tile < c.n) return;
    c.tile = 0;
    if (++c.pr < HR) return;
    c.pr = 0;
    do {
        ++c.b;
    } while (c.b < B && tile_base[c.b + 1] == tile_base[c.b]);
    c.n = c.b < B ? tile_base[c.b + 1] - tile_base[c.b] : 0;
}

// Consumer-group barrier on an mbarrier (bounded, unlike bar.sync).
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &uses) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait_bounded(bar, uses & 1);
    ++uses;
    __syncwarp();
    return ok;
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// The running row max only moves when a tile's max exceeds it by more than
// this many log2 units; until then probabilities stay below 2^8 relative to
// the stale max, which the f32 sums and the bf16 P carry without loss, and
// the final division by the row sum is unchanged.
constexpr float kRescaleThreshold = 8.0f;

template <int NWC, int STAGES>
__global__ void __launch_bounds__((NWC + 1) * 32)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const AttnKParams p) {
    constexpr int NT = (NWC + 1) * 32;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * kStageBytes);
    uint64_t *empty = full + STAGES;
    uint64_t *cbar = empty + STAGES;  // consumer-group barrier
    int *misc = reinterpret_cast<int *>(cbar + 1);  // [0] abort, [1] last flag, [2] c_first, [3] ncontrib
    int *tile_base = misc + 4;                      // [B + 1]
    int *scan_tmp = tile_base + (p.B + 1);          // [NT]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int HR = p.Hkv * p.RG;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWC);
        }
        mbar_init(cbar, NWC);
        misc[0] = 0;
        fence_mbar_init();
    }
    if (tid == NWC * 32) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }

    // ---- tiles per sequence and their prefix sums (every CTA, identically)
    {
        const int per = (p.B + NT - 1) / NT;
        const int b0 = tid * per, b1 = min(p.B, b0 + per);
        int sum = 0;
        for (int b = b0; b < b1; ++b) {
            const int L = p.prefix_lens[b];
            const bool ok = L >= 0 && (long long)L + p.T <= p.S_max;
            sum += ok ? (L + p.T + kBK - 1) / kBK : 0;
        }
        scan_tmp[tid] = sum;
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int i = 0; i < NT; ++i) {
                const int v = scan_tmp[i];
                scan_tmp[i] = acc;
                acc += v;
            }
            tile_base[p.B] = acc;
        }
        __syncthreads();
        int acc = scan_tmp[tid];
        for (int b = b0; b < b1; ++b) {
            tile_base[b] = acc;
            const int L = p.prefix_lens[b];
            const bool ok = L >= 0 && (long long)L + p.T <= p.S_max;
            acc += ok ? (L + p.T + kBK - 1) / kBK : 0;
        }
    }
    // ---- per-sequence status (CTA 0 only): prefix length, then the tree
    if (blockIdx.x == 0 && p.seq_status) {
        for (int b = tid; b < p.B; b += NT) {
            const int L = p.prefix_lens[b];
            p.seq_status[b] = (L >= 0 && (long long)L + p.T <= p.S_max) ? SV_OK : SV_ERR_BAD_INPUT;
        }
        __syncthreads();
        if (p.parents) {
            for (int i = tid; i < p.B * p.T; i += NT) {
                const int b = i / p.T, t = i - b * p.T;
                const int pa = p.parents[i];
                if (t == 0 ? pa != -1 : (pa < 0 || pa >= t)) p.seq_status[b] = SV_ERR_BAD_INPUT;
            }
        }
    }
    __syncthreads();

    // Units are split over min(grid, U) CTAs so that every working CTA holds at
    // least one unit: the merge counts on every CTA in a pair's range arriving.
    const long long U = (long long)tile_base[p.B] * HR;
    const int nctas = (int)(U < (long long)gridDim.x ? U : (long long)gridDim.x);
    if ((int)blockIdx.x >= nctas) return;
    const long long u_begin = cta_begin(U, nctas, blockIdx.x);
    const long long u_end = cta_begin(U, nctas, blockIdx.x + 1);

    volatile int *abort_flag = misc;

    if (warp == NWC) {
        // ================= producer: one elected lane streams K/V tiles
        if (lane == 0) {
            Cursor cur = cursor_at(tile_base, p.B, HR, u_begin);
            long long k = 0;
            for (long long u = u_begin; u < u_end; ++u, ++k) {
                const int s = (int)(k % STAGES);
                const uint32_t ph = (uint32_t)((k / STAGES) & 1);
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                    *abort_flag = 1;
                    if (p.seq_status) p.seq_status[cur.b] = SV_ERR_TIMEOUT;
                    break;
                }
                if (*abort_flag) break;
                const int kvh = cur.pr / p.RG;
                const int y = (cur.b * p.Hkv + kvh) * p.S_max + cur.tile * kBK;
                uint8_t *st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &tmk, 0, y, &full[s]);
                tma_load_2d(st + kBox, &tmk, 64, y, &full[s]);
                tma_load_2d(st + 2 * kBox, &tmv, 0, y, &full[s]);
                tma_load_2d(st + 3 * kBox, &tmv, 64, y, &full[s]);
                cursor_next(cur, tile_base, p.B, HR);
            }
            // drain: every copy issued must land before the CTA may exit
            const long long first = k > STAGES ? k - STAGES : 0;
            for (long long j = first; j < k; ++j)
                mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1));
        }
        return;
    }

    // ===================== consumers: warp `warp` owns 16 query rows
    uint32_t qf[8][4];
    float o[16][4];
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
    uint64_t anc0 = 0, anc1 = 0;
    int L = 0, kv_end = 0, seg_first_tile = 0, kvh = 0, rg = 0;
    bool seg_is_first = true;
    uint32_t cbar_uses = 0;
    const int rsub = lane >> 2;  // row within the 8-row half
    const int csub = lane & 3;
    const float sc = p.scale_log2;
    // Per-thread offsets of this lane's ldmatrix row inside a stage.  With the
    // 128-byte swizzle the 16-byte chunk index is XORed with (row mod 8), and
    // row mod 8 is lane mod 8 for every row this lane addresses.
    uint32_t offK[4], offV[4];
    {
        const int l7 = lane & 7;
        const int kb = (lane >> 4) & 1, cb = (lane >> 3) & 1;  // K: +8 keys, +1 chunk
        const int vb = (lane >> 3) & 1, vc = (lane >> 4) & 1;  // V: +8 keys, +1 chunk
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
            offK[qd] = (uint32_t)((kb * 8 + l7) * 128 + (((2 * qd + cb) ^ l7) << 4));
            offV[qd] = (uint32_t)(2 * kBox + (vb * 8 + l7) * 128 + (((2 * qd + vc) ^ l7) << 4));
        }
    }

    Cursor cur = cursor_at(tile_base, p.B, HR, u_begin);
    long long k = 0;
    for (long long u = u_begin; u < u_end; ++u, ++k) {
        if (u == u_begin || cur.tile == 0) {
            // ---- a new (sequence, KV head, row group) segment
            kvh = cur.pr / p.RG;
            rg = cur.pr - kvh * p.RG;
            L = p.prefix_lens[cur.b];
            kv_end = L + p.T;
            seg_first_tile = cur.tile;
            seg_is_first = (u == u_begin);
            m0 = m1 = kNegInf;
            l0 = l1 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            const int r0 = rg * p.rows_per_rg + warp * 16 + rsub;
            const int r1 = r0 + 8;
            const uint16_t *q0 = nullptr, *q1 = nullptr;
            anc0 = anc1 = 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = half ? r1 : r0;
                if (r >= p.M) continue;
                const int t = r / p.G, g = r - t * p.G;
                const uint16_t *qrow =
                    p.q + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
                uint64_t anc = 0;
                if (p.parents == nullptr) {
                    anc = t >= 63 ? ~0ull : ((1ull << (t + 1)) - 1ull);
                } else {
                    int nd = t;
                    for (int step = 0; step < kMaxT && nd >= 0; ++step) {
                        anc |= 1ull << nd;
                        const int pn = p.parents[(size_t)cur.b * p.T + nd];
                        if (pn >= nd) break;
                        nd = pn;
                    }
                }
                if (half) {
                    q1 = qrow;
                    anc1 = anc;
                } else {
                    q0 = qrow;
                    anc0 = anc;
                }
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int c0 = 16 * kk + 2 * csub;
                qf[kk][0] = q0 ? ld_u32(q0 + c0) : 0u;
                qf[kk][1] = q1 ? ld_u32(q1 + c0) : 0u;
                qf[kk][2] = q0 ? ld_u32(q0 + c0 + 8) : 0u;
                qf[kk][3] = q1 ? ld_u32(q1 + c0 + 8) : 0u;
            }
        }

        const int s = (int)(k % STAGES);
        const uint32_t ph = (uint32_t)((k / STAGES) & 1);
        bool ok = mbar_wait_bounded(&full[s], ph);
        if (!ok || *abort_flag) {
            *abort_flag = 1;
            if (p.seq_status) p.seq_status[cur.b] = SV_ERR_TIMEOUT;
            break;
        }
        const uint32_t st_base = base_u32 + s * kStageBytes;
        const int kbase = cur.tile * kBK;

        // ---- S = Q K^T over 64 keys
        float sacc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t rowK = st_base + offK[kk & 3] + (kk >> 2) * kBox;
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(rowK + jp * 2048, b0, b1, b2, b3);
                mma_bf16_16816(sacc[2 * jp], qf[kk], b0, b1);
                mma_bf16_16816(sacc[2 * jp + 1], qf[kk], b2, b3);
            }
        }

        // ---- mask: only tiles reaching the new rows or the sequence end
        if (kbase + kBK > L) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = kbase + 8 * j + 2 * csub + (e & 1);
                    const uint64_t anc = e < 2 ? anc0 : anc1;
                    const bool allowed =
                        key < L || (key < kv_end && ((anc >> (unsigned)(key - L)) & 1ull));
                    if (!allowed) sacc[j][e] = kNegInf;
                }
            }
        }

        // ---- online softmax in the log2 domain, max moved lazily
        float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mx0 = fmaxf(mx0, fmaxf(sacc[j][0], sacc[j][1]));
            mx1 = fmaxf(mx1, fmaxf(sacc[j][2], sacc[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float c0 = mx0 * sc, c1 = mx1 * sc;   // raw max -> log2 units
        const bool up0 = c0 > m0 + kRescaleThreshold;
        const bool up1 = c1 > m1 + kRescaleThreshold;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float a0 = up0 ? ex2_approx(m0 - c0) : 1.f;
            const float a1 = up1 ? ex2_approx(m1 - c1) : 1.f;
            if (up0) m0 = c0;
            if (up1) m1 = c1;
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                o[j][0] *= a0;
                o[j][1] *= a0;
                o[j][2] *= a1;
                o[j][3] *= a1;
            }
        }
        const float nb0 = m0 == kNegInf ? 0.f : -m0;
        const float nb1 = m1 == kNegInf ? 0.f : -m1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sacc[j][0] = ex2_approx(fmaf(sacc[j][0], sc, nb0));
            sacc[j][1] = ex2_approx(fmaf(sacc[j][1], sc, nb0));
            sacc[j][2] = ex2_approx(fmaf(sacc[j][2], sc, nb1));
            sacc[j][3] = ex2_approx(fmaf(sacc[j][3], sc, nb1));
            l0 += sacc[j][0] + sacc[j][1];
            l1 += sacc[j][2] + sacc[j][3];
        }

        // ---- O += P V over 64 keys
        const bool need_vfix = kbase + kBK > kv_end;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
            pa[1] = pack_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
            pa[2] = pack_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
            pa[3] = pack_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
            if (!need_vfix) {
#pragma unroll
                for (int djp = 0; djp < 8; ++djp) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(st_base + offV[djp & 3] + (djp >> 2) * kBox + kk * 2048, v0, v1,
                              v2, v3);
                    mma_bf16_16816(o[2 * djp], pa, v0, v1);
                    mma_bf16_16816(o[2 * djp + 1], pa, v2, v3);
                }
            } else {  // rows past the sequence's last slot may hold anything: zero them
                const int k0 = kbase + 16 * kk + 2 * csub;
                const uint32_t mlo =
                    (k0 < kv_end ? 0x0000ffffu : 0u) | (k0 + 1 < kv_end ? 0xffff0000u : 0u);
                const uint32_t mhi =
                    (k0 + 8 < kv_end ? 0x0000ffffu : 0u) | (k0 + 9 < kv_end ? 0xffff0000u : 0u);
#pragma unroll
                for (int djp = 0; djp < 8; ++djp) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(st_base + offV[djp & 3] + (djp >> 2) * kBox + kk * 2048, v0, v1,
                              v2, v3);
                    mma_bf16_16816(o[2 * djp], pa, v0 & mlo, v1 & mhi);
                    mma_bf16_16816(o[2 * djp + 1], pa, v2 & mlo, v3 & mhi);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // ---- end of a segment: write the rows, or a partial to be merged
        if (cur.tile == cur.n - 1 || u == u_end - 1) {
            float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
            float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
            lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
            const int rr0 = warp * 16 + rsub, rr1 = rr0 + 8;  // rows within the row group
            const int r0 = rg * p.rows_per_rg + rr0, r1 = rg * p.rows_per_rg + rr1;
            const bool whole = seg_first_tile == 0 && cur.tile == cur.n - 1;
            if (whole) {
                const float i0 = 1.f / lt0, i1 = 1.f / lt1;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = half ? r1 : r0;
                    if (r >= p.M) continue;
                    const int t = r / p.G, g = r - t * p.G;
                    uint16_t *orow =
                        p.out + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
                    const float inv = half ? i1 : i0;
#pragma unroll
                    for (int dj = 0; dj < 16; ++dj) {
                        const uint32_t pk = pack_bf16x2(o[dj][2 * half] * inv, o[dj][2 * half + 1] * inv);
                        *reinterpret_cast<uint32_t *>(orow + 8 * dj + 2 * csub) = pk;
                    }
                }
            } else {
                const int slot = seg_is_first ? 0 : 1;
                float *po = p.part_o + ((size_t)blockIdx.x * 2 + slot) * p.rows_per_rg * kD;
                float *pml = p.part_ml + ((size_t)blockIdx.x * 2 + slot) * p.rows_per_rg * 2;
#pragma unroll
                for (int dj = 0; dj < 16; ++dj) {
                    *reinterpret_cast<float2 *>(po + (size_t)rr0 * kD + 8 * dj + 2 * csub) =
                        make_float2(o[dj][0], o[dj][1]);
                    *reinterpret_cast<float2 *>(po + (size_t)rr1 * kD + 8 * dj + 2 * csub) =
                        make_float2(o[dj][2], o[dj][3]);
                }
                if (csub == 0) {
                    *reinterpret_cast<float2 *>(pml + rr0 * 2) = make_float2(m0, lt0);
                    *reinterpret_cast<float2 *>(pml + rr1 * 2) = make_float2(m1, lt1);
                }
                __threadfence();
                const int pair = (cur.b * p.Hkv + kvh) * p.RG + rg;
                const long long ub = (long long)tile_base[cur.b] * HR + (long long)cur.pr * cur.n;
                const int c_first = cta_of(U, nctas, ub);
                const int c_last = cta_of(U, nctas, ub + cur.n - 1);
                if (!group_sync(cbar, cbar_uses)) {
                    *abort_flag = 1;
                    if (p.seq_status) p.seq_status[cur.b] = SV_ERR_TIMEOUT;
                    break;
                }
                if (warp == 0 && lane == 0) {
                    __threadfence();
                    const int old = atomicAdd(&p.counters[pair], 1);
                    misc[1] = (old == c_last - c_first) ? 1 : 0;
                }
                if (!group_sync(cbar, cbar_uses)) {
                    *abort_flag = 1;
                    if (p.seq_status) p.seq_status[cur.b] = SV_ERR_TIMEOUT;
                    break;
                }
                const bool last = misc[1] != 0;
                if (last) {
                    __threadfence();
                    // merge every contributor's partial for this warp's 16 rows
                    for (int i = 0; i < 16; ++i) {
                        const int rr = warp * 16 + i;
                        const int r = rg * p.rows_per_rg + rr;
                        if (r >= p.M) break;
                        float mstar = kNegInf;
                        for (int c = c_first; c <= c_last; ++c) {
                            const int sl = cta_begin(U, nctas, c) >= ub ? 0 : 1;
                            const float mc = __ldcg(p.part_ml + ((size_t)c * 2 + sl) * p.rows_per_rg * 2 + rr * 2);
                            mstar = fmaxf(mstar, mc);
                        }
                        float lsum = 0.f;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int c = c_first; c <= c_last; ++c) {
                            const int sl = cta_begin(U, nctas, c) >= ub ? 0 : 1;
                            const size_t slot_i = (size_t)c * 2 + sl;
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
                                p.part_ml + slot_i * p.rows_per_rg * 2 + rr * 2));
                            const float wgt = ml.x == kNegInf ? 0.f : exp2f(ml.x - mstar);
                            lsum += ml.y * wgt;
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                p.part_o + (slot_i * p.rows_per_rg + rr) * kD + lane * 4));
                            acc.x += v.x * wgt;
                            acc.y += v.y * wgt;
                            acc.z += v.z * wgt;
                            acc.w += v.w * wgt;
                        }
                        const float inv = 1.f / lsum;
                        const int t = r / p.G, g = r - t * p.G;
                        uint16_t *orow =
                            p.out + (((size_t)cur.b * p.T + t) * p.Hq + kvh * p.G + g) * kD;
                        uint2 pk;
                        pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                        pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                        *reinterpret_cast<uint2 *>(orow + lane * 4) = pk;
                    }
                    if (warp == 0 && lane == 0) p.counters[pair] = 0;  // ready for the next call
                }
            }
        }
        cursor_next(cur, tile_base, p.B, HR);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D view [rows = B*Hkv*S_max, D] of a bf16 cache, 64x64 boxes, 128-byte swizzle.
static bool make_cache_map(CUtensorMap *map, const void *base, long long rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBK};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

typedef void (*AttnKernelFn)(const CUtensorMap, const CUtensorMap, const AttnKParams);

struct KernelEntry {
    int nwc;
    int stages;
    const void *fn;
};

template <int NWC, int STAGES>
static KernelEntry entry() {
    return KernelEntry{NWC, STAGES, reinterpret_cast<const void *>(&tree_attention_kernel<NWC, STAGES>)};
}

static const KernelEntry *kernel_for(int nwc) {
    static const KernelEntry table[] = {entry<1, 3>(), entry<2, 3>(), entry<3, 3>(), entry<4, 3>(),
                                        entry<6, 4>(), entry<8, 4>()};
    for (const KernelEntry &e : table)
        if (e.nwc >= nwc) return &e;
    return nullptr;
}

static int smem_bytes(int stages, int nwc, int B) {
    return stages * kStageBytes + 1024 + (2 * stages + 1) * 8 + 16 + (B + 1) * 4 + (nwc + 1) * 32 * 4;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Occupancy of one kernel on one device for a given shared-memory size,
// queried once and cached: these runtime queries cost far more than a launch
// and would otherwise make short calls host-bound.
static int cached_occupancy(const KernelEntry &e, int smem, int *sms_out) {
    struct Entry {
        int dev;
        const void *fn;
        int smem, occ, sms;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].fn == e.fn && cache[i].smem == smem) {
            *sms_out = cache[i].sms;
            return cache[i].occ;
        }
    const int threads = (e.nwc + 1) * 32;
    if (cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes(e.stages, e.nwc, kMaxB)) != cudaSuccess)
        return -1;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, e.fn, threads, smem) != cudaSuccess)
        return -1;
    const int sms = device_sm_count();
    if (sms <= 0 || occ < 1) return -1;
    if (ncache < 64) cache[ncache++] = Entry{dev, e.fn, smem, occ, sms};
    *sms_out = sms;
    return occ;
}

sv_status plan_attention(int B, int T, int Hq, int Hkv, int D, AttnPlan *plan) {
    if (D != kD || T > kMaxT || B > kMaxB) return SV_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    const int M = G * T;
    if (M > 512) return SV_ERR_UNSUPPORTED;
    int nwc = (M + 15) / 16;
    int rg = 1;
    if (nwc > 8) {
        rg = (nwc + 7) / 8;
        nwc = 8;
    }
    const KernelEntry *e = kernel_for(nwc);
    if (!e) return SV_ERR_UNSUPPORTED;
    AttnPlan pl{};
    pl.nwc = e->nwc;
    pl.stages = e->stages;
    pl.rows_per_rg = 16 * pl.nwc;
    pl.rg = rg;
    pl.smem = smem_bytes(pl.stages, pl.nwc, B);
    int sms = 0;
    const int occ = cached_occupancy(*e, pl.smem, &sms);
    if (occ < 1) return SV_ERR_CUDA;
    pl.grid = sms * occ;
    size_t off = 0;
    pl.off_counters = off;
    off = align_up(off + sizeof(int) * (size_t)B * Hkv * rg, 256);
    pl.off_part_o = off;
    off = align_up(off + sizeof(float) * (size_t)pl.grid * 2 * pl.rows_per_rg * kD, 256);
    pl.off_part_ml = off;
    off = align_up(off + sizeof(float) * (size_t)pl.grid * 2 * pl.rows_per_rg * 2, 256);
    pl.bytes = off;
    *plan = pl;
    return SV_OK;
}

sv_status launch_tree_attention(const AttnArgs &a, const AttnPlan &pl, void *ws,
                                cudaStream_t st) {
    const long long rows = (long long)a.B * a.Hkv * a.S_max;
    CUtensorMap tmk, tmv;
    if (!make_cache_map(&tmk, a.k, rows) || !make_cache_map(&tmv, a.v, rows)) return SV_ERR_CUDA;
    AttnKParams p{};
    p.q = static_cast<const uint16_t *>(a.q);
    p.out = static_cast<uint16_t *>(a.out);
    p.prefix_lens = a.prefix_lens;
    p.parents = a.parents;
    p.seq_status = a.seq_status;
    p.B = a.B;
    p.T = a.T;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.S_max = a.S_max;
    p.M = p.G * a.T;
    p.RG = pl.rg;
    p.rows_per_rg = pl.rows_per_rg;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    char *base = static_cast<char *>(ws);
    p.counters = reinterpret_cast<int *>(base + pl.off_counters);
    p.part_o = reinterpret_cast<float *>(base + pl.off_part_o);
    p.part_ml = reinterpret_cast<float *>(base + pl.off_part_ml);
    const KernelEntry *e = kernel_for(pl.nwc);
    const int threads = (pl.nwc + 1) * 32;
    void *args[] = {&tmk, &tmv, &p};
    if (cudaLaunchKernel(e->fn, dim3(pl.grid), dim3(threads), args, pl.smem, st) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

}  // namespace sv
