// sv_noalloc.cu -- chain verify for callers that cannot allocate device memory.
//
// spec_verify_chain needs a caller-provided workspace for its fastest small-batch
// kernel.  Some callers have no way to provide one: code running inside a runtime
// that owns every device allocation (a serving engine's arena, a plugin interface
// that hands out only input and output buffers), or a hot path where an allocation
// call is not allowed.  spec_verify_chain_noalloc takes the same inputs and outputs
// and uses a scratch array that lives in this library's own device image instead.
//
// The scratch is a file-scope __device__ array of NOALLOC_SCRATCH_BYTES.  In host
// code its name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current, and the
// array is zeroed then; the kernel leaves the parts that must start at zero (the
// per-row arrival counters) zeroed again at the end of every call.
#include <mutex>

#include "spec_verify.h"
#include "sv_internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)256 << 10;  // 256 KiB, held by every device that loads the library
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void* g_scratch_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device (set up on first use).
sv_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return SV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
        if (cudaMemset(p, 0, NOALLOC_SCRATCH_BYTES) != cudaSuccess) return SV_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return SV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SV_OK;
}

}  // namespace

extern "C" {

sv_status spec_verify_chain_noalloc(const void* target_logits, sv_dtype tdt, const void* draft, sv_dtype ddt,
                                    sv_draft_kind dk, const int32_t* draft_tokens, const float* temperature, int B,
                                    int K, int V, uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                    int32_t* out_count, float* out_accept_prob, void* stream) {
    // the argument checks of spec_verify_chain, before anything touches the device
    if (B < 0 || K < 0 || V < 1) return SV_ERR_INVALID_ARG;
    const size_t need = spec_verify_workspace_size(B, K, V);
    if (B > 0 && need == 0) return SV_ERR_INVALID_ARG;  // K or V beyond the library's limits
    if ((unsigned)tdt > 1u || (unsigned)ddt > 1u || (unsigned)dk > 1u) return SV_ERR_INVALID_ARG;
    if (dk == SV_DRAFT_PROBS && ddt != SV_F32) return SV_ERR_INVALID_ARG;
    if (need > NOALLOC_SCRATCH_BYTES) return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!target_logits || !temperature || !out_tokens || !out_count || (K > 0 && (!draft_tokens || !draft)))
        return SV_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const sv_status st = scratch_for_current_device(&scratch);
    if (st != SV_OK) return st;
    return sv::chain_with_scratch(target_logits, tdt, draft, ddt, dk, draft_tokens, temperature, B, K, V, seed,
                                  offset, out_tokens, out_count, out_accept_prob, scratch, NOALLOC_SCRATCH_BYTES,
                                  stream);
}

}  // extern "C"
