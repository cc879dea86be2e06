// sv_host.cu -- chain verify from host memory: one packed copy in, the verify, one copy
// out, all enqueued on the caller's stream (include/spec_verify.h).
#include <cstdint>

#include "spec_verify.h"
#include "sv_internal.h"

namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" {

sv_status spec_verify_host_sizes(int B, int K, int V, sv_dtype tdt, sv_dtype ddt, sv_draft_kind dk,
                                 size_t* offsets, size_t* in_bytes, size_t* out_bytes) {
    if (B < 0 || B > 65535 || K < 0 || K > 64 || V < 1 || V > (1 << 24)) return SV_ERR_INVALID_ARG;
    if ((unsigned)tdt > 1u || (unsigned)ddt > 1u || (unsigned)dk > 1u) return SV_ERR_INVALID_ARG;
    if (dk == SV_DRAFT_PROBS && ddt != SV_F32) return SV_ERR_INVALID_ARG;
    const size_t tsz = tdt == SV_BF16 ? 2 : 4, dsz = ddt == SV_BF16 ? 2 : 4;
    size_t off[4];
    off[0] = 0;
    off[1] = round256(off[0] + (size_t)B * (K + 1) * V * tsz);
    off[2] = round256(off[1] + (size_t)B * K * V * dsz);
    off[3] = round256(off[2] + (size_t)B * K * 4);
    const size_t total = round256(off[3] + (size_t)B * 4);
    if (offsets)
        for (int i = 0; i < 4; ++i) offsets[i] = off[i];
    if (in_bytes) *in_bytes = total;
    if (out_bytes) *out_bytes = (size_t)B * (K + 2) * 4;
    return SV_OK;
}

sv_status spec_verify_chain_host(const void* h_in, void* d_in, void* h_out, void* d_out, sv_dtype tdt, sv_dtype ddt,
                                 sv_draft_kind dk, int B, int K, int V, uint64_t seed, uint64_t offset,
                                 void* workspace, size_t ws_bytes, void* stream) {
    size_t off[4], in_bytes = 0, out_bytes = 0;
    const sv_status st = spec_verify_host_sizes(B, K, V, tdt, ddt, dk, off, &in_bytes, &out_bytes);
    if (st != SV_OK) return st;
    if (B == 0) return SV_OK;
    if (!h_in || !d_in || !h_out || !d_out) return SV_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return sv::launch_status(e);
    unsigned char* base = static_cast<unsigned char*>(d_in);
    int32_t* out_tokens = static_cast<int32_t*>(d_out);
    int32_t* out_count = out_tokens + (size_t)B * (K + 1);
    const sv_status v = spec_verify_chain(base + off[0], tdt, base + off[1], ddt, dk,
                                          reinterpret_cast<const int32_t*>(base + off[2]),
                                          reinterpret_cast<const float*>(base + off[3]), B, K, V, seed, offset,
                                          out_tokens, out_count, nullptr, workspace, ws_bytes, stream);
    if (v != SV_OK) return v;
    e = cudaMemcpyAsync(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return sv::launch_status(e);
    return SV_OK;
}

}  // extern "C"
