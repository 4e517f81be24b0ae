// sv_compact.cu -- compaction of the accepted path's K/V rows.
//
// The enlarged KV cache of tree verification holds one row per candidate
// node ("Parallel Decoding" glossary, "Limites du parallel decoding"); after
// acceptance the accepted path becomes the committed continuation and the
// rest is discarded ("Chapitre 9 -- Décodage spéculatif" §9.1).  Row
// L + path[d] moves to row L + d for d = 0..a, in place.
//
// One CTA per sequence.  The path increases strictly, so path[d] >= d: the
// destination slot L + d of position d is never the source of a LATER
// position.  The moves, one per (position, KV head) pair in order of d, go in
// rounds of consecutive pairs, every head at once: a round reads all its rows
// (K and V) into registers before any of them is written back, so a source
// is always read before a move of an earlier round could have overwritten it.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kCT = 256;
constexpr int kCompactRegs = 8;        // 16-byte words a thread holds in a round
constexpr int kMaxRoundPairs = 256;    // (position, head) pairs per round
constexpr int kMaxRowVecs = 32;        // 16-byte words per row: D <= 256 bf16

__global__ void __launch_bounds__(kCT) compact_kv_kernel(CompactArgs a) {
    __shared__ size_t s_src_off[kMaxRoundPairs], s_dst_off[kMaxRoundPairs];
    __shared__ unsigned char s_move[kMaxRoundPairs];
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x;
    const int L = a.prefix_lens[b];
    const int acc = a.accepted_len[b];
    const int vpr = a.D / 8;  // 16-byte words per row
    __syncthreads();          // every thread has read L before new_kv_lens (may alias) is written

    if (acc < 0) {
        if (threadIdx.x == 0) {
            a.new_kv_lens[b] = L;
            if (a.seq_status) a.seq_status[b] = SV_OK;
        }
        return;
    }
    int bad = (L < 0) || ((long long)L + acc + 1 > a.S_max) ||
              (a.path_nodes != nullptr && acc >= a.path_stride);
    // a paged cache: the page of a slot must exist
    auto page_ok = [&](int slot) {
        const int pg = a.block_table[(size_t)b * a.max_pages + slot / a.page_size];
        return pg >= 0 && pg < a.num_pages;
    };
    if (!bad && a.path_nodes) {
        const int32_t *path = a.path_nodes + (size_t)b * a.path_stride;
        for (int d = threadIdx.x; d <= acc; d += kCT) {
            const int src = path[d];
            if (d == 0 ? src != 0 : src <= path[d - 1]) bad = 1;
            if ((long long)L + src >= a.S_max) bad = 1;
            if (!bad && a.block_table && (!page_ok(L + src) || !page_ok(L + d))) bad = 1;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (threadIdx.x == 0) {
            a.new_kv_lens[b] = L;
            if (a.seq_status) a.seq_status[b] = SV_ERR_BAD_INPUT;
        }
        return;
    }
    if (a.path_nodes && acc > 0) {
        const int32_t *path = a.path_nodes + (size_t)b * a.path_stride;
        uint4 *kc = static_cast<uint4 *>(a.k);
        uint4 *vc = static_cast<uint4 *>(a.v);
        // offset (16-byte words) of row `slot` of KV head h: contiguous
        // [B, Hkv, S_max, D], or through the page table
        auto row_off = [&](int h, int slot) -> size_t {
            if (!a.block_table) return (((size_t)b * a.Hkv + h) * a.S_max + slot) * vpr;
            const int pg = a.block_table[(size_t)b * a.max_pages + slot / a.page_size];
            return (((size_t)pg * a.Hkv + h) * a.page_size + slot % a.page_size) * vpr;
        };
        const int per_pair = 2 * vpr;  // K and V words of one row
        const int npairs = acc * a.Hkv;  // positions 1..acc (the root never moves) x heads
        const int round = min(kMaxRoundPairs, kCT * kCompactRegs / per_pair);
        for (int q0 = 0; q0 < npairs; q0 += round) {
            const int np = min(round, npairs - q0);
            for (int i = threadIdx.x; i < np; i += kCT) {
                const int q = q0 + i, d = 1 + q / a.Hkv, h = q - (d - 1) * a.Hkv;
                const int src = path[d];
                s_move[i] = src != d;
                s_src_off[i] = row_off(h, L + src);
                s_dst_off[i] = row_off(h, L + d);
            }
            __syncthreads();
            const int items = np * per_pair;
            uint4 reg[kCompactRegs];
#pragma unroll
            for (int k = 0; k < kCompactRegs; ++k) {
                const int it = threadIdx.x + k * kCT;
                if (it < items) {
                    const int pr = it / per_pair, rem = it - pr * per_pair;
                    const int kv = rem >= vpr, w = rem - kv * vpr;
                    if (s_move[pr]) reg[k] = (kv ? vc : kc)[s_src_off[pr] + w];
                }
            }
            __syncthreads();  // every source of the round is read
#pragma unroll
            for (int k = 0; k < kCompactRegs; ++k) {
                const int it = threadIdx.x + k * kCT;
                if (it < items) {
                    const int pr = it / per_pair, rem = it - pr * per_pair;
                    const int kv = rem >= vpr, w = rem - kv * vpr;
                    if (s_move[pr]) (kv ? vc : kc)[s_dst_off[pr] + w] = reg[k];
                }
            }
            __syncthreads();  // before the next round's offsets replace these
        }
    }
    if (threadIdx.x == 0) {
        a.new_kv_lens[b] = L + acc + 1;
        if (a.seq_status) a.seq_status[b] = SV_OK;
    }
}

sv_status launch_compact_kv(const CompactArgs &a, cudaStream_t st) {
    if (a.D % 8 != 0 || a.D / 8 > kMaxRowVecs) return SV_ERR_UNSUPPORTED;
    CompactArgs ka = a;
    void *args[] = {&ka};
    return launch_pdl((const void *)compact_kv_kernel, dim3(a.B), dim3(kCT), 0, st, args) ==
                   cudaSuccess
               ? SV_OK
               : SV_ERR_CUDA;
}

}  // namespace sv
