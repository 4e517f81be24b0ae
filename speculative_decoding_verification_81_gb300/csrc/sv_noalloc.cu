// sv_noalloc.cu -- sv_verify_chain_noalloc: chain acceptance for callers that
// cannot allocate device memory where they call the library (see the header
// for who they are).  The scratch that sv_verify_chain takes from a caller
// workspace lives here instead, in one fixed array of the library.
#include <cstdint>
#include <mutex>

#include "sv_internal.h"

namespace {

// The library's own scratch: SV_NOALLOC_SCRATCH_BYTES on every device that
// loads the library, held until the process exits.  In host code this name
// is a host-side stand-in, not a device address: kernels get the address
// that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached for the process: valid in
// the device's primary context until a cudaDeviceReset of the device.
sv_status scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return SV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" sv_status sv_verify_chain_noalloc(const void *target_logits, const void *draft_logits,
                                             sv_dtype dtype, const int32_t *draft_tokens,
                                             const float *u_accept, const float *u_sample, int B,
                                             int N, int V, int32_t *accepted_len,
                                             int32_t *out_tokens, float *probs_out,
                                             int32_t *seq_status, sv_stream_t stream) {
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample ||
        !accepted_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || V <= 0) return SV_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SV_ERR_INVALID_ARG;
    if (N > 63 || V >= (1 << 30)) return SV_ERR_UNSUPPORTED;
    const sv::VocabPlan pl = sv::plan_vocab(true, B, N, V, dtype);
    if ((size_t)B * pl.rows_per_seq * pl.nchunks >= (1u << 31)) return SV_ERR_UNSUPPORTED;
    if (pl.bytes > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;  // beyond the fixed array

    void *scratch = nullptr;
    const sv_status st = scratch_on_current_device(&scratch);
    if (st != SV_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the counters (arrivals, the timeout flag) must start at zero; everything
    // else is written before it is read
    if (cudaMemsetAsync(static_cast<char *>(scratch) + pl.off_counters, 0,
                        sizeof(int) * (2 * (size_t)B + 4), s) != cudaSuccess)
        return SV_ERR_CUDA;
    sv::ChainArgs a{target_logits, draft_logits, draft_tokens, nullptr, u_accept, u_sample, B, N, V,
                    accepted_len, out_tokens, probs_out, seq_status};
    return sv::launch_verify_chain(a, dtype, pl, scratch, s);
}
