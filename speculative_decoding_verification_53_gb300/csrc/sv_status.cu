// sv_status.cu -- row-status summary of a finished verify call (include/spec_verify.h).
//
// Every verify entry reports problems per batch row and goes on with the other rows:
// out_count[b] = 0 for bad data (NaN or +inf in a row the rule read, a row with no
// finite logit, an out-of-range token, a malformed tree), out_count[b] = -1 where a
// bounded device-side wait gave up.  spec_verify_count_invalid counts the first kind
// and spec_verify_rows_status summarises both into the call's status, on the device
// and in stream order after the call, so a caller reads a few bytes instead of
// copying every count back.
#include <cstdint>

#include "spec_verify.h"
#include "sv_common.cuh"
#include "sv_internal.h"

namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountMaxB = 1 << 24;

// One CTA: strided counts per thread of the rows with count 0 and with count -1, then
// warp and block sums.  status = 0: out[0] = the count-0 rows; status = 1: out[0] = the
// call's sv_status, out[1] = count-0 rows, out[2] = count -1 rows.  Written once (the
// output needs no initialisation).
__global__ void __launch_bounds__(kCountThreads) count_rows_kernel(const int32_t* count, int B, int32_t* out,
                                                                   int status) {
    __shared__ int s_warp[2][kCountThreads / 32];
    sv::pdl_trigger();
    sv::pdl_wait();  // the verify kernel that wrote the counts has completed
    int n0 = 0, nt = 0;
    for (int i = (int)threadIdx.x; i < B; i += kCountThreads) {
        const int c = count[i];
        n0 += c == 0 ? 1 : 0;
        nt += c == sv::SV_COUNT_TIMEOUT ? 1 : 0;
    }
    n0 = __reduce_add_sync(0xffffffffu, n0);
    nt = __reduce_add_sync(0xffffffffu, nt);
    if ((threadIdx.x & 31) == 0) {
        s_warp[0][threadIdx.x >> 5] = n0;
        s_warp[1][threadIdx.x >> 5] = nt;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int a = __reduce_add_sync(0xffffffffu, s_warp[0][threadIdx.x]);
        const int t = __reduce_add_sync(0xffffffffu, s_warp[1][threadIdx.x]);
        if (threadIdx.x == 0) {
            if (status) {
                out[0] = t > 0 ? (int32_t)SV_ERR_TIMEOUT : (a > 0 ? (int32_t)SV_ERR_BAD_INPUT : (int32_t)SV_OK);
                out[1] = a;
                out[2] = t;
            } else {
                out[0] = a;
            }
        }
    }
}

sv_status launch_count(const int32_t* out_count, int B, int32_t* out, int status, void* stream) {
    if (B < 0 || B > kCountMaxB || !out || (B > 0 && !out_count)) return SV_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kCountThreads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return sv::launch_status(cudaLaunchKernelEx(&cfg, count_rows_kernel, out_count, B, out, status));
}

}  // namespace

extern "C" {

sv_status spec_verify_count_invalid(const int32_t* out_count, int B, int32_t* out_invalid, void* stream) {
    return launch_count(out_count, B, out_invalid, 0, stream);
}

sv_status spec_verify_rows_status(const int32_t* out_count, int B, int32_t* out_status, void* stream) {
    return launch_count(out_count, B, out_status, 1, stream);
}

}  // extern "C"
