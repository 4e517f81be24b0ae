// sv_attention.cu -- host side of the verification attention: TMA tensor
// maps over the K/V caches and Q, the launch plan (grid, pipeline depth,
// shared memory, workspace) and the launch of the tcgen05 kernel in
// sv_attention_tc.cu.
#include <mutex>

#include "sv_attn_common.cuh"
#include "sv_internal.h"

namespace sv {

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

// 2-D view [rows, D] of a bf16 cache (rows = B*Hkv*S_max, or num_pages*Hkv*page_size
// for a paged one), boxes of 64 dims x box_rows rows, 128-byte swizzle.
static bool make_cache_map(CUtensorMap *map, const void *base, long long rows, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [B*T nodes][Hq heads][D] of Q; a box is 64 dims of G heads of
// `nodes` consecutive nodes, i.e. the rows (t, g) of one row group in the
// order t*G + g, 128-byte swizzle.  Nodes past B*T read as zeros.
static bool make_q_map(CUtensorMap *map, const void *q, int B, int T, int Hq, int G, int nodes) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hq, (cuuint64_t)B * T};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hq * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)nodes};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
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
static int cached_occupancy(const void *fn, int threads, int max_smem, int smem, int *sms_out) {
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
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem) {
            *sms_out = cache[i].sms;
            return cache[i].occ;
        }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
        cudaSuccess)
        return -1;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess)
        return -1;
    const int sms = device_sm_count();
    if (sms <= 0 || occ < 1) return -1;
    if (ncache < 64) cache[ncache++] = Entry{dev, fn, smem, occ, sms};
    *sms_out = sms;
    return occ;
}

// Largest number of clusters of `cs` CTAs of the attention kernel that the
// current device keeps resident at once (0 if none), cached like the occupancy.
static int cached_max_clusters(const void *fn, int smem, int cs) {
    struct Entry {
        int dev;
        const void *fn;
        int smem, cs, n;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem && cache[i].cs == cs)
            return cache[i].n;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    cudaGetLastError();  // a refused query leaves no error behind
    if (ncache < 64) cache[ncache++] = Entry{dev, fn, smem, cs, n};
    return n;
}

static void plan_workspace(AttnPlan &pl, int B, int Hkv) {
    size_t off = 0;
    pl.off_pair_ctr = off;  // [pair][arrived, ready][softmax warp]
    off = align_up(off + sizeof(int) * (size_t)B * Hkv * pl.rg * 2 * kSoftmaxWarps, 256);
    pl.off_part_o = off;
    off = align_up(off + sizeof(float) * (size_t)pl.grid * 2 * pl.mrows * kD, 256);
    pl.off_part_ml = off;
    off = align_up(off + sizeof(float) * (size_t)pl.grid * 2 * pl.mrows * 4, 256);
    pl.bytes = off;
}

sv_status plan_attention(int B, int T, int Hq, int Hkv, int D, int S_max, AttnPlan *plan,
                         int max_ctas) {
    if (D != kD || T > kMaxT || B > kMaxB) return SV_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    const int M = G * T;
    if (M > 512 || G > 128) return SV_ERR_UNSUPPORTED;
    AttnPlan pl{};
    pl.mrows = M <= 64 ? 64 : 128;  // M=64 products for small row groups
    // a row group holds whole nodes (G rows each), so that its Q rows are one box
    pl.rows_per_rg = pl.mrows - pl.mrows % G;
    pl.rg = (M + pl.rows_per_rg - 1) / pl.rows_per_rg;
    // three K/V stages when shared memory allows, else two
    int max_optin = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return SV_ERR_CUDA;
    pl.stages = tc_smem_bytes(3, pl.mrows, B) <= max_optin ? 3 : 2;
    pl.smem = tc_smem_bytes(pl.stages, pl.mrows, B);
    if (pl.smem > max_optin) return SV_ERR_UNSUPPORTED;
    int sms = 0;
    const int occ = cached_occupancy(tc_kernel_fn(pl.stages, pl.mrows), kTcThreads, max_optin,
                                     pl.smem, &sms);
    if (occ < 1) return SV_ERR_CUDA;
    pl.grid = sms * occ;
    pl.cluster = 1;
    plan_workspace(pl, B, Hkv);  // sized for the whole device's flat split, whichever mode runs
    if (max_ctas > 0 && max_ctas < pl.grid) pl.grid = max_ctas;
    // Few row groups (fewer than half the CTAs the device holds): one cluster
    // per group, its tiles shared by the cluster's CTAs and merged in
    // distributed shared memory, instead of a flat split whose groups straddle
    // CTAs and merge through global memory.  The largest cluster size whose
    // clusters the device keeps resident all at once, up to the tiles a group
    // can have.
    const long long groups = (long long)B * Hkv * pl.rg;
    const int max_tiles = (S_max + kBK - 1) / kBK;
    if (groups * 2 <= pl.grid) {
        for (int cs = kMaxCluster; cs >= 2; cs >>= 1) {
            if (cs > max_tiles || groups * cs > pl.grid) continue;
            if (cached_max_clusters(tc_kernel_fn(pl.stages, pl.mrows), pl.smem, cs) >= groups) {
                pl.cluster = cs;
                pl.grid = (int)(groups * cs);
                break;
            }
        }
    }
    *plan = pl;
    return SV_OK;
}

sv_status launch_tree_attention(const AttnArgs &a, const AttnPlan &pl, void *ws,
                                cudaStream_t st) {
    const bool paged = a.block_table != nullptr;
    const long long rows = paged ? (long long)a.num_pages * a.Hkv * a.page_size
                                 : (long long)a.B * a.Hkv * a.S_max;
    const int box_rows = paged && a.page_size < kBK ? a.page_size : kBK;
    CUtensorMap tmk, tmv, tmq;
    const int G = a.Hq / a.Hkv;
    if (!make_cache_map(&tmk, a.k, rows, box_rows) || !make_cache_map(&tmv, a.v, rows, box_rows) ||
        !make_q_map(&tmq, a.q, a.B, a.T, a.Hq, G, pl.rows_per_rg / G))
        return SV_ERR_CUDA;
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
    p.pair_ctr = reinterpret_cast<int *>(base + pl.off_pair_ctr);
    p.part_o = reinterpret_cast<float *>(base + pl.off_part_o);
    p.part_ml = reinterpret_cast<float *>(base + pl.off_part_ml);
    p.block_table = a.block_table;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.page_size = a.page_size;
    p.node_counts = a.node_counts;
    p.node_count_add = a.node_count_add;
    p.cluster = pl.cluster;
    p.hook = a.hook;
    p.hook_acc = a.hook_acc;
    p.hook_path = a.hook_path;
    p.hook_path_stride = a.hook_path_stride;
    void *args[] = {&tmk, &tmv, &tmq, &p};
    const void *fn = tc_kernel_fn(pl.stages, pl.mrows);
    if (pl.cluster <= 1)
        return launch_pdl(fn, dim3(pl.grid), dim3(kTcThreads), pl.smem, st, args) == cudaSuccess
                   ? SV_OK
                   : SV_ERR_CUDA;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)pl.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv
