// sv_api.cu -- the C ABI declared in include/spec_verify.h: argument checks on the
// host, launch-shape choice, dispatch to the kernels.  Nothing here allocates.
#include <cstdlib>
#include <string>

#include "spec_verify.h"
#include "sv_internal.h"

namespace sv {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

sv_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return SV_OK;
    g_last_cuda_error = e;
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
}

}  // namespace sv

using sv::g_last_cuda_error;
using sv::launch_status;

namespace {

constexpr int kMaxK = 64;
constexpr int kMaxNodes = 1024;
constexpr int kMaxDepth = 64;
constexpr int kMaxV = 1 << 24;
constexpr int kMaxB = 65535;

// Launch-shape override for tuning: SPEC_VERIFY_CLUSTER in {1, 2, 4, 8, 16}.
int cluster_override() {
    static const int v = [] {  // read once (thread-safe initialisation)
        const char* s = std::getenv("SPEC_VERIFY_CLUSTER");
        const int x = s ? std::atoi(s) : 0;
        return (x == 1 || x == 2 || x == 4 || x == 8 || x == 16) ? x : 0;
    }();
    return v;
}

bool is_dtype(int d) { return d == SV_F32 || d == SV_BF16; }

struct DeviceInfo {
    int sms = 0;
    int major = 0;
};

// SM count and compute capability of the current device (queried on every call:
// cheap, and correct when the caller switches devices).
sv_status device_info(DeviceInfo& info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&info.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return launch_status(e);
    if (info.major < 10) return SV_ERR_UNSUPPORTED;  // built for sm_103a (thread-block clusters, DSMEM)
    return SV_OK;
}

// Kernel-family override for comparison runs and tests: SPEC_VERIFY_PATH =
// "spec" (position-parallel), "staged" (shared-memory staging), "stream"
// (register streaming), "eager" (all positions staged at once), "ring" (ring-streamed
// walk); anything else picks automatically.
enum PathChoice { PATH_AUTO = 0, PATH_SPEC = 1, PATH_STAGED = 2, PATH_STREAM = 3, PATH_EAGER = 4, PATH_RING = 5 };

int path_override() {
    static const int v = [] {  // read once (thread-safe initialisation)
        const char* s = std::getenv("SPEC_VERIFY_PATH");
        int r = PATH_AUTO;
        if (s) {
            const std::string p(s);
            if (p == "spec") r = PATH_SPEC;
            if (p == "staged") r = PATH_STAGED;
            if (p == "stream") r = PATH_STREAM;
            if (p == "eager") r = PATH_EAGER;
            if (p == "ring") r = PATH_RING;
        }
        return r;
    }();
    return v;
}

// Test hook for the timeout path (SPEC_VERIFY_TEST_STALL=<row>): in the shared-memory
// staged walk, batch row <row> announces its first copy without issuing it, so its
// bounded wait runs out after 50 us and the row reports out_count = -1.  Off (-1) unless
// the variable is set; read once.
int stall_row_override() {
    static const int v = [] {
        const char* s = std::getenv("SPEC_VERIFY_TEST_STALL");
        return s ? std::atoi(s) : -1;
    }();
    return v;
}

size_t dtype_size(int d) { return d == SV_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t round16(size_t x) { return (x + 15) & ~(size_t)15; }

// Staging layout for a chain launch, or nslot = 0 when the staged kernel does not apply
// (rows not 16-byte aligned, or one slot does not fit in shared memory).
sv::StageLayout chain_stage_layout(const void* target, int tdt, const void* draft, int ddt, int dk, bool uses_draft,
                                   int B, int K, int V, int G, int num_sms) {
    sv::StageLayout L{0, 0, 0, 0, 0, 0};
    const size_t tsz = dtype_size(tdt), dsz = dk == SV_DRAFT_PROBS ? 4 : dtype_size(ddt);
    if (!aligned16(target) || (V * tsz) % 16) return L;
    if (uses_draft && (!aligned16(draft) || (V * dsz) % 16)) return L;
    const size_t nvec = (V + 7) / 8, cmax = ((nvec + G - 1) / G) * 8;
    const size_t t_bytes = round16(cmax * tsz);
    const bool small = (long long)B * G <= num_sms;  // one CTA per SM or fewer: prefetch positions ahead
    // Large batches keep only the target chunk on chip and stream the draft-logit row from
    // global memory (its statistics while the target chunk lands, its second read for the
    // draw from L2): half the shared memory per row, so twice the rows in flight.
    // Measured at B = 256, K = 8, V = 152064, T = 0.7 (clusters of 8): see the kernel.
    const bool d_direct = !small && uses_draft && dk == SV_DRAFT_LOGITS;
    const size_t d_bytes = (uses_draft && dk == SV_DRAFT_LOGITS && !d_direct) ? round16(cmax * dsz) : 0;
    const size_t probs = (uses_draft && dk == SV_DRAFT_PROBS) ? round16(cmax * 4) : 0;
    const size_t fixed = sv::STAGE_HEADER + probs + sv::draw_smem_bytes(V, G) + 64;
    const size_t budget = small ? (size_t)sv::MAX_DYN_SMEM - 8192 : (size_t)100 * 1024;
    const size_t slot = t_bytes + d_bytes;
    if (fixed + slot > budget) return L;
    size_t nslot = small ? (budget - fixed) / slot : 1;
    if (nslot > (size_t)K + 1) nslot = K + 1;
    if (nslot > 16) nslot = 16;
    L.nslot = (int)nslot;
    L.slot_bytes = (int)slot;
    L.t_bytes = (int)t_bytes;
    L.probs_bytes = (int)probs;
    L.prefetch_l2 = small ? 1 : 0;
    L.d_direct = d_direct ? 1 : 0;
    return L;
}

// Cluster size of the position-parallel kernel, or 0 where the walking kernels are
// faster:
//  - one CTA per SM when the batch allows a cluster of at least 4: the largest power of
//    two (at most 16) with B (K + 1) G <= SMs;
//  - else a cluster that leaves each CTA 12 K to 24 K elements (G >= 2), when the
//    launch fits in two waves of CTAs (how many fit on an SM set by the kernel's shared
//    memory, at most four).  Measured against the staged walk, K = 5: V = 32000 at G = 2,
//    B = 16 / 32 / 64: 10.5 / 11.4 / 17.4 us against 16.5 / 18.3 / 20.1; V = 128256 at
//    G = 8, B = 8 / 16: 11.5 / 17.6 against 16.7 / 21.2; at B = 128 (3.4 waves) 29.7
//    against 28.2.  Where it runs, every position is read, the rejected ones included.
//  forced: the kernel was requested (SPEC_VERIFY_PATH=spec, the allocation-free entry);
//  the one-CTA-per-SM size is used when the rules above give none.
int spec_cluster(int B, int K, int V, int tsz, int dsz, int num_sms, bool forced) {
    int G = 16;
    while (G > 1 && (long long)B * (K + 1) * G > num_sms) G >>= 1;
    if (G >= 4) return G;
    int Gc = 1;
    while (Gc < 16 && (long long)V >= 2LL * Gc * 12288) Gc *= 2;
    if (Gc >= 2) {
        const size_t smem = sv::spec_smem_bytes(V, Gc, tsz, dsz, nullptr, nullptr) + 8192;  // + static, reserved
        long long fit = (long long)(232448 / smem);
        if (fit > 4) fit = 4;
        if (fit >= 1 && (long long)B * (K + 1) * Gc <= 2LL * fit * num_sms) return Gc;
    }
    return forced ? G : 0;
}

// Cluster size of the ring-streamed walk (sv_chain_ring.cu), or 0 where it is not the
// kernel to take.  It is made for batches too large to stage on chip: clusters of 4
// CTAs of 128 threads (each CTA at least one full 2048-element stage of the row), taken
// when B clusters fill the SMs at least twice over, so that every row is resident
// while HBM streams.  forced (SPEC_VERIFY_PATH=ring): any batch, a cluster of 4, or of
// SPEC_VERIFY_CLUSTER (2, 4 or 8) when set.
int ring_cluster(int B, int V, int num_sms, bool forced) {
    int G = 4;
    const int o = cluster_override();
    if (forced && (o == 1 || o == 2 || o == 4 || o == 8)) G = o;
    if (forced) {
        while (G > 1 && V < G * 8) G >>= 1;  // every CTA owns part of the row
        return G;
    }
    (void)B;
    (void)num_sms;
    return 0;  // measured slower than the staged walk on every batch tried (only when forced)
}

// Stage layout of the ring-streamed walk: three stages of 2048 elements of the target
// row and of the draft row (logits, or fp32 probabilities for the draw).
sv::RingLayout chain_ring_layout(int tdt, int ddt, int dk, bool uses_draft) {
    sv::RingLayout R{3, 0, 0};
    R.t_bytes = (int)round16((size_t)2048 * dtype_size(tdt));
    const size_t d = uses_draft ? round16((size_t)2048 * (dk == SV_DRAFT_PROBS ? 4 : dtype_size(ddt))) : 0;
    R.stage_bytes = R.t_bytes + (int)d;
    return R;
}

// Kernel choice for a chain launch:
//  - position-parallel (sv_chain_spec.cu) for small and moderate batches when a workspace
//    is given (spec_cluster): every position of every row at once, the latency of one
//    position instead of K+1, at the price of reading the positions after the first
//    rejection;
//  - ring-streamed walk (sv_chain_ring.cu) for large batches of aligned rows (ring_cluster);
//  - shared-memory staged walk (sv_chain_staged.cu) when rows are 16-byte aligned;
//  - register-streaming walk (sv_chain.cu) otherwise.
sv_status run_chain(const sv::ChainArgs& a, int tdt, int ddt, int dk, bool uses_draft, int num_sms, void* ws,
                    size_t ws_bytes, cudaStream_t stream, int forced_path = PATH_AUTO) {
    const int path = forced_path != PATH_AUTO ? forced_path : path_override();
    const size_t tsz = dtype_size(tdt), dsz = dk == SV_DRAFT_PROBS ? 4 : dtype_size(ddt);
    const bool aligned = aligned16(a.target) && (a.V * tsz) % 16 == 0 &&
                         (!uses_draft || (aligned16(a.draft) && (a.V * dsz) % 16 == 0));
    // all positions staged at once, one cluster per row (only when requested: measured slower
    // than the position-parallel kernel at B = 1, 14.2 against 9.4 us)
    if (path == PATH_EAGER && aligned && a.K + 1 <= 16) {
        int Ge = 16;
        while (Ge > 1 && (long long)a.B * Ge > num_sms) Ge >>= 1;
        {
            const cudaError_t e = sv::launch_chain_eager(a, tdt, ddt, dk, Ge, stream);
            if (e == cudaSuccess) return SV_OK;
            if (e != cudaErrorInvalidClusterSize) return launch_status(e);
            (void)cudaGetLastError();
        }
    }
    if ((path == PATH_AUTO || path == PATH_SPEC) && aligned && ws && ((uintptr_t)ws & 255u) == 0 &&
        a.K + 1 <= sv::SPEC_MAX_POS) {
        const int Gs = spec_cluster(a.B, a.K, a.V, (int)tsz, (int)dsz, num_sms, path == PATH_SPEC);
        if (Gs > 0 && ws_bytes >= sv::spec_workspace_bytes(a.B, a.K, a.V, Gs)) {
            const cudaError_t e = sv::launch_chain_spec(a, ws, tdt, ddt, dk, Gs, stream);
            if (e == cudaSuccess) return SV_OK;
            if (e != cudaErrorInvalidClusterSize) return launch_status(e);
            (void)cudaGetLastError();
        }
    }
    if ((path == PATH_AUTO || path == PATH_RING) && aligned) {
        const int Gr = ring_cluster(a.B, a.V, num_sms, path == PATH_RING);
        if (Gr > 0) {
            const cudaError_t e =
                sv::launch_chain_ring(a, chain_ring_layout(tdt, ddt, dk, uses_draft), tdt, ddt, dk, Gr, stream);
            if (e == cudaSuccess) return SV_OK;
            if (e != cudaErrorInvalidClusterSize) return launch_status(e);
            (void)cudaGetLastError();
        }
    }
    const int G = sv::choose_cluster(a.B, a.V, num_sms);
    const sv::StageLayout L = chain_stage_layout(a.target, tdt, a.draft, ddt, dk, uses_draft, a.B, a.K, a.V, G, num_sms);
    if (L.nslot > 0 && path != PATH_STREAM) {
        sv::ChainArgs as = a;
        as.stall_row = stall_row_override();
        as.stall_ns = 50000u;
        const cudaError_t e = sv::launch_chain_staged(as, L, tdt, ddt, dk, G, stream);
        if (e == cudaSuccess) return SV_OK;
        if (e != cudaErrorInvalidClusterSize) return launch_status(e);
        (void)cudaGetLastError();
    }
    return launch_status(sv::launch_chain(a, tdt, ddt, dk, G, stream));
}


}  // namespace

namespace sv {

sv_status chain_with_scratch(const void* target_logits, int tdt, const void* draft, int ddt, int dk,
                             const int32_t* draft_tokens, const float* temperature, int B, int K, int V,
                             uint64_t seed, uint64_t offset, int32_t* out_tokens, int32_t* out_count,
                             float* out_accept_prob, void* scratch, size_t scratch_bytes, void* stream) {
    // same checks and the same kernel choice as spec_verify_chain, with the scratch as
    // the workspace: the position-parallel kernel (the one that uses it) where the
    // automatic rule picks it, the kernels that need no scratch elsewhere
    if (B < 0 || B > kMaxB || K < 0 || K > kMaxK || V < 1 || V > kMaxV) return SV_ERR_INVALID_ARG;
    if (!is_dtype(tdt) || !is_dtype(ddt)) return SV_ERR_INVALID_ARG;
    if (dk != SV_DRAFT_PROBS && dk != SV_DRAFT_LOGITS) return SV_ERR_INVALID_ARG;
    if (dk == SV_DRAFT_PROBS && ddt != SV_F32) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !temperature || !out_tokens || !out_count || (K > 0 && (!draft_tokens || !draft)))
        return SV_ERR_INVALID_ARG;
    DeviceInfo info;
    sv_status st = device_info(info);
    if (st != SV_OK) return st;
    ChainArgs a{target_logits, draft, draft_tokens, temperature, B, K, V, seed, offset,
                out_tokens, out_count, out_accept_prob};
    return run_chain(a, tdt, ddt, dk, K > 0, info.sms, scratch, scratch_bytes, (cudaStream_t)stream);
}

int choose_cluster(int B, int V, int num_sms) {
    const int forced = cluster_override();
    if (forced) return forced;
    // As many CTAs per row as keep at least 2048 elements each (at most 16), while the
    // grid stays within about 16 CTAs per SM: rows are walked position by position, so a
    // wide split shortens each row's serial chain and many rows in flight hide latency.
    int G = 1;
    while (G < 16 && V / (2 * G) >= 2048 && (long long)B * 2 * G <= 16LL * num_sms) G *= 2;
    return G;
}

}  // namespace sv

extern "C" {

size_t spec_verify_workspace_size(int B, int K, int V) {
    if (B < 0 || K < 0 || K > kMaxK || V < 1 || V > kMaxV) return 0;
    size_t need = 0;
    for (int G = 1; G <= 16; G *= 2) {
        const size_t b = sv::spec_workspace_bytes(B, K, V, G);
        if (b > need) need = b;
    }
    return need;
}

sv_status spec_verify_chain(const void* target_logits, sv_dtype tdt, const void* draft, sv_dtype ddt,
                            sv_draft_kind dk, const int32_t* draft_tokens, const float* temperature, int B, int K,
                            int V, uint64_t seed, uint64_t offset, int32_t* out_tokens, int32_t* out_count,
                            float* out_accept_prob, void* workspace, size_t ws_bytes, void* stream) {
    if (B < 0 || B > kMaxB || K < 0 || K > kMaxK || V < 1 || V > kMaxV) return SV_ERR_INVALID_ARG;
    if (!is_dtype(tdt) || !is_dtype(ddt)) return SV_ERR_INVALID_ARG;
    if (dk != SV_DRAFT_PROBS && dk != SV_DRAFT_LOGITS) return SV_ERR_INVALID_ARG;
    if (dk == SV_DRAFT_PROBS && ddt != SV_F32) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !temperature || !out_tokens || !out_count || (K > 0 && (!draft_tokens || !draft)))
        return SV_ERR_INVALID_ARG;
    DeviceInfo info;
    sv_status st = device_info(info);
    if (st != SV_OK) return st;
    sv::ChainArgs a{target_logits, draft, draft_tokens, temperature, B, K, V, seed, offset,
                    out_tokens, out_count, out_accept_prob};
    return run_chain(a, tdt, ddt, dk, K > 0, info.sms, workspace, ws_bytes, (cudaStream_t)stream);
}

sv_status spec_sample_and_verify(const void* target_logits, sv_dtype tdt, const void* draft_logits, sv_dtype ddt,
                                 const float* temperature, int B, int K, int V, uint64_t seed, uint64_t offset,
                                 int32_t* out_draft_tokens, int32_t* out_tokens, int32_t* out_count,
                                 float* out_accept_prob, void* workspace, size_t ws_bytes, void* stream) {
    if (B < 0 || B > kMaxB || K < 0 || K > kMaxK || V < 1 || V > kMaxV) return SV_ERR_INVALID_ARG;
    if (!is_dtype(tdt) || !is_dtype(ddt)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !temperature || !out_tokens || !out_count || (K > 0 && (!draft_logits || !out_draft_tokens)))
        return SV_ERR_INVALID_ARG;
    DeviceInfo info;
    sv_status st = device_info(info);
    if (st != SV_OK) return st;
    if (K > 0) {
        const sv::SampleArgs s{draft_logits, temperature, B, K, V, seed, offset, out_draft_tokens};
        const cudaError_t e = sv::launch_draft_sample(s, ddt, info.sms, (cudaStream_t)stream);
        if (e != cudaSuccess) return launch_status(e);
    }
    // the verify reads the tokens the sampling kernel wrote (same stream, so in order)
    const sv::ChainArgs a{target_logits, draft_logits, out_draft_tokens, temperature, B, K, V, seed, offset,
                          out_tokens, out_count, out_accept_prob};
    return run_chain(a, tdt, ddt, SV_DRAFT_LOGITS, K > 0, info.sms, workspace, ws_bytes, (cudaStream_t)stream);
}

sv_status spec_greedy_accept(const void* target_logits, sv_dtype tdt, const int32_t* draft_tokens, int B, int K,
                             int V, int32_t* out_tokens, int32_t* out_count, void* stream) {
    if (B < 0 || B > kMaxB || K < 0 || K > kMaxK || V < 1 || V > kMaxV) return SV_ERR_INVALID_ARG;
    if (!is_dtype(tdt)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !out_tokens || !out_count || (K > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
    DeviceInfo info;
    sv_status st = device_info(info);
    if (st != SV_OK) return st;
    sv::ChainArgs a{target_logits, nullptr, draft_tokens, nullptr, B, K, V, 0, 0, out_tokens, out_count, nullptr};
    // the draft kind and dtype do not matter for greedy rows; use the smallest instantiation
    return run_chain(a, tdt, SV_F32, SV_DRAFT_PROBS, false, info.sms, nullptr, 0, (cudaStream_t)stream);
}

sv_status spec_verify_tree(const void* target_logits, sv_dtype tdt, const void* draft, sv_dtype ddt,
                           sv_draft_kind dk, const int32_t* node_tokens, const int32_t* parent,
                           const float* temperature, int B, int N, int V, int max_depth, uint64_t seed,
                           uint64_t offset, int32_t* out_tokens, int32_t* out_count, int32_t* out_path,
                           void* stream) {
    return spec_verify_tree_rule(target_logits, tdt, draft, ddt, dk, node_tokens, parent, temperature, B, N, V,
                                 max_depth, SV_SIBLINGS_WITHOUT_REPLACEMENT, seed, offset, out_tokens, out_count,
                                 out_path, stream);
}

sv_status spec_verify_tree_rule(const void* target_logits, sv_dtype tdt, const void* draft, sv_dtype ddt,
                                sv_draft_kind dk, const int32_t* node_tokens, const int32_t* parent,
                                const float* temperature, int B, int N, int V, int max_depth,
                                sv_sibling_rule sibling_rule, uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                int32_t* out_count, int32_t* out_path, void* stream) {
    if (B < 0 || B > kMaxB || N < 1 || N > kMaxNodes || V < 1 || V > kMaxV || max_depth < 1 ||
        max_depth > kMaxDepth)
        return SV_ERR_INVALID_ARG;
    if (sibling_rule != SV_SIBLINGS_WITHOUT_REPLACEMENT && sibling_rule != SV_SIBLINGS_IID)
        return SV_ERR_INVALID_ARG;
    if (!is_dtype(tdt) || !is_dtype(ddt)) return SV_ERR_INVALID_ARG;
    if (dk != SV_DRAFT_PROBS && dk != SV_DRAFT_LOGITS) return SV_ERR_INVALID_ARG;
    if (dk == SV_DRAFT_PROBS && ddt != SV_F32) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !draft || !node_tokens || !parent || !temperature || !out_tokens || !out_count ||
        !out_path)
        return SV_ERR_INVALID_ARG;
    DeviceInfo info;
    sv_status st = device_info(info);
    if (st != SV_OK) return st;
    sv::TreeArgs a{target_logits, draft, node_tokens, parent, temperature, B, N, V, max_depth, seed, offset,
                   out_tokens, out_count, out_path, (int)sibling_rule};
    const int G = sv::choose_cluster(B, V, info.sms);
    // shared-memory staged walk (with the children's rows prefetched) when rows are aligned
    const size_t tsz = dtype_size(tdt), dsz = dk == SV_DRAFT_PROBS ? 4 : dtype_size(ddt);
    if (path_override() != PATH_STREAM && aligned16(target_logits) && aligned16(draft) && (V * tsz) % 16 == 0 &&
        (V * dsz) % 16 == 0) {
        const size_t nvec = (V + 7) / 8, cmax = ((nvec + G - 1) / G) * 8;
        sv::StageLayout L{0, 0, 0, 0, 0, 0};
        L.t_bytes = (int)round16(cmax * tsz);
        L.slot_bytes = L.t_bytes + (int)round16(cmax * dsz);
        const bool small = (long long)B * G <= info.sms;
        // two CTAs a SM for a large batch (about 8 KB of static shared memory each)
        const size_t budget = small ? (size_t)sv::MAX_DYN_SMEM - 16 * 1024 : (size_t)104 * 1024;
        const size_t fixed = sv::STAGE_HEADER + sv::tree_array_bytes(N) + sv::tree_work_bytes(V, G) +
                             sv::draw_smem_bytes(V, G);
        if (fixed + L.slot_bytes <= budget) {
            size_t nslot = (budget - fixed) / L.slot_bytes;
            if (nslot > 16) nslot = 16;
            if (!small && nslot > 2) nslot = 2;
            L.nslot = (int)nslot;
            const cudaError_t e = sv::launch_tree_staged(a, L, tdt, ddt, dk, G, (cudaStream_t)stream);
            if (e == cudaSuccess) return SV_OK;
            if (e != cudaErrorInvalidClusterSize) return launch_status(e);
            (void)cudaGetLastError();
        }
    }
    return launch_status(sv::launch_tree(a, tdt, ddt, dk, G, (cudaStream_t)stream));
}

const char* spec_verify_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

const char* spec_verify_status_string(sv_status status) {
    switch (status) {
        case SV_OK: return "SV_OK: success";
        case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: a size, pointer, dtype or kind argument is invalid";
        case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: outside what the library handles";
        case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA runtime call or kernel launch failed";
        case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded device-side wait gave up";
        case SV_ERR_BAD_INPUT: return "SV_ERR_BAD_INPUT: invalid data in a batch row";
    }
    return "unknown sv_status";
}

}  // extern "C"
