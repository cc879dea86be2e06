// sv_status.cu -- data-error summary of a finished verify call (include/spec_verify.h).
//
// Every verify entry reports bad data per batch row, as out_count[b] = 0 (NaN or
// +inf in a row the rule read, a row with no finite logit, an out-of-range token, a
// malformed tree), and goes on with the other rows.  spec_verify_count_invalid
// counts those rows on the device, in stream order after the call, so a caller can
// turn them into the call's SV_ERR_BAD_INPUT status with one 4-byte read instead of
// copying every count back.
#include <cstdint>

#include "spec_verify.h"
#include "sv_common.cuh"
#include "sv_internal.h"

namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountMaxB = 1 << 24;

// One CTA: a strided count per thread, then warp and block sums; the single result
// is written once (the output needs no initialisation).
__global__ void __launch_bounds__(kCountThreads) count_invalid_kernel(const int32_t* count, int B, int32_t* out) {
    __shared__ int s_warp[kCountThreads / 32];
    sv::pdl_trigger();
    sv::pdl_wait();  // the verify kernel that wrote the counts has completed
    int n = 0;
    for (int i = (int)threadIdx.x; i < B; i += kCountThreads) n += count[i] == 0 ? 1 : 0;
    n = __reduce_add_sync(0xffffffffu, n);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = n;
    __syncthreads();
    if (threadIdx.x < 32) {
        int v = s_warp[threadIdx.x];
        v = __reduce_add_sync(0xffffffffu, v);
        if (threadIdx.x == 0) *out = v;
    }
}

}  // namespace

extern "C" {

sv_status spec_verify_count_invalid(const int32_t* out_count, int B, int32_t* out_invalid, void* stream) {
    if (B < 0 || B > kCountMaxB || !out_invalid || (B > 0 && !out_count)) return SV_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kCountThreads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return sv::launch_status(cudaLaunchKernelEx(&cfg, count_invalid_kernel, out_count, B, out_invalid));
}

}  // extern "C"
