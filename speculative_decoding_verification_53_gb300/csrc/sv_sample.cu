// sv_sample.cu -- the draft tokens of a round drawn on the GPU, ahead of the verify.
//
// "[논문 리뷰] Fast Inference from Transformers via Speculative Decoding", section 2,
// Step 1: the draft model proposes x_1..x_K by sampling from its own distribution.
// When the draft's K distributions are known at once (heads that predict several
// positions from one hidden state), the proposals and the verify can be one call:
// x_k is the inverse-CDF draw of the word-2 Philox uniform of slot k from
// q_k = softmax(draft_k / T), or argmax(draft_k) for a greedy row, and the chain
// verify then runs on those tokens (sv_api.cu).
//
// One G-CTA cluster per (batch row, position).  When the draft rows are 16-byte aligned
// each CTA brings its chunk of the row into shared memory with one bulk copy, reduces
// it to (max, sum) or (max, argmax) there, combines with the cluster through
// distributed shared memory and runs the split inverse-CDF search on the staged chunk;
// other rows are streamed from global memory with the same steps.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

template <int DDT>
struct QWeights {  // w_i = q_i = exp2((d_i - m) c) / S
    static constexpr int kTilesInFlight = 4;  // global loads: several in flight per lane
    const void* drow;
    float c, m, inv_s;
    bool al;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float d[VEC];
        load8<DDT>(drow, e0, hi, al, neg_inf(), d);
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[j] = ex2((d[j] - m) * c) * inv_s;
    }
};

template <int DDT>
__global__ void __launch_bounds__(NT) draft_sample_kernel(const SampleArgs a) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    extern __shared__ float tile_sum[];
    __shared__ BlockScratch sc;
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)
    const int g = (int)cluster_rank(), G = (int)cluster_size();
    const int k = (int)blockIdx.y, b = (int)blockIdx.z;
    const int V = a.V;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const size_t dsz = DDT == DT_BF16 ? 2 : 4;
    const void* drow = (const char*)a.draft + ((size_t)b * a.K + k) * (size_t)V * dsz;
    const bool al = ((uintptr_t)drow & 15) == 0;
    const float T = a.temperature[b];
    const bool greedy = !(T > 0.f);
    int32_t* out = a.out_draft_tokens + (size_t)b * a.K + k;
    int phase = 0;
    if (greedy) {
        ArgMax am = thread_argmax<DDT>(drow, lo, hi, al);
        am = cluster_argmax(am, sc, phase);
        const bool bad = am.bad || !(am.v > neg_inf()) || am.v == pos_inf();
        if (g == 0 && threadIdx.x == 0) *out = bad ? -1 : am.i;
    } else {
        const float c = LOG2E / T;
        const float u = slot_draft_uniform(a.seed, a.offset, (uint64_t)b, (uint64_t)k);
        LSE ds = thread_lse<DDT>(drow, lo, hi, al, c);
        LSE none{neg_inf(), 0.f, 0};
        cluster_lse2(ds, none, c, sc, phase);
        const bool bad = ds.bad || !(ds.m > neg_inf()) || ds.m == pos_inf();
        if (bad) {
            if (g == 0 && threadIdx.x == 0) *out = -1;
        } else {
            const QWeights<DDT> qw{drow, c, ds.m, 1.f / ds.s, al};
            const DrawResult d = cluster_draw(qw, lo, hi, u, tile_sum, sc, phase);
            if (d.owner < 0 || d.failed) {
                if (g == 0 && threadIdx.x == 0) *out = -1;
            } else if (g == d.owner && threadIdx.x == 0) {
                *out = d.token;
            }
        }
    }
    // No trailing cluster barrier: peers only ever push into this CTA's inbox, and the
    // last exchange (the same sequence in every CTA of the cluster) completed on this
    // CTA's own barrier, so nothing is written into its shared memory any more.
}

template <int DDT>
__global__ void __launch_bounds__(NT) draft_sample_staged_kernel(const SampleArgs a, int chunk_bytes) {
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(dsm);
    unsigned char* db = dsm + STAGE_HEADER;
    float* tile_sum = reinterpret_cast<float*>(db + chunk_bytes);
    __shared__ BlockScratch sc;
    __shared__ float s_u;
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)
    const int g = (int)cluster_rank(), G = (int)cluster_size();
    const int k = (int)blockIdx.y, b = (int)blockIdx.z;
    const int V = a.V;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    constexpr int dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* drow = reinterpret_cast<const unsigned char*>(a.draft) + ((size_t)b * a.K + k) * V * dsz;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 32) s_u = slot_draft_uniform(a.seed, a.offset, (uint64_t)b, (uint64_t)k);
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)n * dsz);
        if (n) bulk_g2s(db, drow + (size_t)lo * dsz, (uint32_t)n * dsz, bar);
    }
    const float T = a.temperature[b];
    const bool greedy = !(T > 0.f);
    int32_t* out = a.out_draft_tokens + (size_t)b * a.K + k;
    __syncthreads();  // the barrier is initialised (by thread 0) before anyone polls it
    const int fail = __syncthreads_or(threadIdx.x == 0 && !mbar_wait_bounded(bar, 0));  // thread 0 polls
    int phase = 0;
    if (greedy) {
        ArgMax am = smem_thread_argmax<DDT>(db, n, lo);
        if (fail) am.bad = 1;
        am = cluster_argmax(am, sc, phase);
        const bool bad = am.bad || !(am.v > neg_inf()) || am.v == pos_inf();
        if (g == 0 && threadIdx.x == 0) *out = bad ? -1 : am.i;
    } else {
        const float c = LOG2E / T;
        LSE ds = smem_thread_lse<DDT>(db, n, c);
        if (fail) ds.bad = 1;
        const PosStats ps = cluster_pos_stats<false>(ds, LSE{neg_inf(), 0.f, 0}, c, 0.f, 0.f, 0, sc, phase);
        if (row_bad_s(ps.t)) {
            if (g == 0 && threadIdx.x == 0) *out = -1;
        } else {
            const StagedP<DDT> qw{db, lo, c, ps.t.m, 1.f / ps.t.s};
            const DrawResult d = cluster_draw(qw, lo, hi, s_u, tile_sum, sc, phase);
            if (d.owner < 0 || d.failed) {
                if (g == 0 && threadIdx.x == 0) *out = -1;
            } else if (g == d.owner && threadIdx.x == 0) {
                *out = d.token;
            }
        }
    }
    // No trailing cluster barrier: peers only ever push into this CTA's inbox, and the
    // last exchange (the same sequence in every CTA of the cluster) completed on this
    // CTA's own barrier, so nothing is written into its shared memory any more.
}

// Cluster size: the largest power of two (at most 16, at least 2048 entries a CTA)
// for which all B * K clusters are resident at once (one wave), else 1.
template <int DDT>
static cudaError_t sample_cluster(long long BK, int V, int& G_out) {
    auto kern = draft_sample_kernel<DDT>;
    static KernelLaunchCache cache;
    int G = 1;
    for (int i = 4; i >= 1; --i) {
        const int g = 1 << i;
        if (V / g < 2048) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(NT, 1, 1);
        cfg.dynamicSmemBytes = draw_smem_bytes(V, g);
        int resident = 0;  // clusters of g CTAs co-resident on the current device
        if (cache.active_clusters((const void*)kern, cfg, g, &resident) != cudaSuccess) {
            (void)cudaGetLastError();
            resident = 0;
        }
        if (resident > 0 && BK <= resident) {
            G = g;
            break;
        }
    }
    G_out = G;
    return cudaSuccess;
}

template <int DDT>
static cudaError_t launch_sample_t(const SampleArgs& a, cudaStream_t stream) {
    auto kern = draft_sample_kernel<DDT>;
    static KernelLaunchCache cache;
    int G = 1;
    cudaError_t e = sample_cluster<DDT>((long long)a.B * a.K, a.V, G);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    // a cluster size whose draw tile sums fit in shared memory (very large rows need G > 1)
    e = cache.pick_cluster((const void*)kern, cfg, G, [&](int g) { return draw_smem_bytes(a.V, g); }, &G);
    if (e != cudaSuccess) return e;
    if (G == 0) return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)G, (unsigned)a.K, (unsigned)a.B);
    cfg.dynamicSmemBytes = draw_smem_bytes(a.V, G);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Staged launch: the cluster is wide enough for a chunk of at most 96 KB, and wider
// still (up to 16, chunks of at least 2048 entries) while B * K * G stays within the SMs.
template <int DDT>
static cudaError_t launch_sample_staged_t(const SampleArgs& a, int num_sms, cudaStream_t stream) {
    auto kern = draft_sample_staged_kernel<DDT>;
    constexpr int dsz = DDT == DT_BF16 ? 2 : 4;
    static KernelLaunchCache cache;
    int max_dyn = 0;
    {
        const cudaError_t e = cache.setup((const void*)kern, &max_dyn);
        if (e != cudaSuccess) return e;
    }
    auto chunk_bytes = [&](int G) {
        const size_t nvec = (size_t)(a.V + VEC - 1) / VEC, cmax = ((nvec + G - 1) / G) * VEC;
        return (cmax * dsz + 15) & ~(size_t)15;
    };
    int G = 1;
    while (G < 16 && chunk_bytes(G) > 96 * 1024) G *= 2;
    while (G < 16 && a.V / (2 * G) >= 2048 && (long long)a.B * a.K * 2 * G <= num_sms) G *= 2;
    size_t cb = chunk_bytes(G);
    size_t smem = STAGE_HEADER + cb + draw_smem_bytes(a.V, G);
    if (smem > (size_t)max_dyn) return cudaErrorInvalidClusterSize;  // the streaming kernel takes it
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    cfg.dynamicSmemBytes = smem;
    int maxc = 0;  // largest cluster the device co-schedules at this shared-memory size
    cudaError_t e = cache.max_cluster((const void*)kern, cfg, &maxc);
    if (e != cudaSuccess) return e;
    if (maxc < G) {
        while (G > 1 && G > maxc) G >>= 1;
        cb = chunk_bytes(G);
        smem = STAGE_HEADER + cb + draw_smem_bytes(a.V, G);
        if (smem > (size_t)max_dyn) return cudaErrorInvalidClusterSize;
        cfg.dynamicSmemBytes = smem;
    }
    cfg.gridDim = dim3((unsigned)G, (unsigned)a.K, (unsigned)a.B);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, (int)cb);
}

cudaError_t launch_draft_sample(const SampleArgs& a, int ddt, int num_sms, cudaStream_t stream) {
    const size_t dsz = ddt == DT_BF16 ? 2 : 4;
    if (((uintptr_t)a.draft & 15) == 0 && ((size_t)a.V * dsz) % 16 == 0) {
        const cudaError_t e = ddt == DT_BF16 ? launch_sample_staged_t<DT_BF16>(a, num_sms, stream)
                                             : launch_sample_staged_t<DT_F32>(a, num_sms, stream);
        if (e != cudaErrorInvalidClusterSize) return e;
        (void)cudaGetLastError();
    }
    if (ddt == DT_BF16) return launch_sample_t<DT_BF16>(a, stream);
    return launch_sample_t<DT_F32>(a, stream);
}

}  // namespace sv
