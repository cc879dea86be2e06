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
// One G-CTA cluster per (batch row, position): the CTAs stream their chunks of the
// draft row to (max, sum) or (max, argmax), combine them through distributed shared
// memory and split the inverse-CDF search the same way as the replacement draw.
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

template <int DDT>
struct QWeights {  // w_i = q_i = exp2((d_i - m) c) / S
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
    extern __shared__ float tile_sum[];
    __shared__ BlockScratch sc;
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
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}

// Cluster size: the largest power of two (at most 16, at least 2048 entries a CTA)
// that keeps the B * K clusters within about 16 CTAs per SM.
static int sample_cluster(int BK, int V, int num_sms) {
    int G = 1;
    while (G < 16 && V / (2 * G) >= 2048 && (long long)BK * 2 * G <= 16LL * num_sms) G *= 2;
    return G;
}

template <int DDT>
static cudaError_t launch_sample_t(const SampleArgs& a, int num_sms, cudaStream_t stream) {
    auto kern = draft_sample_kernel<DDT>;
    static int max_cluster = 0;  // largest cluster the device co-schedules for this kernel
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    if (max_cluster == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(MAX_CLUSTER, 1, 1);
        cfg.dynamicSmemBytes = draw_smem_bytes(a.V, 1);
        int m = 0;
        e = cudaOccupancyMaxPotentialClusterSize(&m, kern, &cfg);
        if (e != cudaSuccess) return e;
        max_cluster = m < 1 ? 1 : m;
    }
    int G = sample_cluster(a.B * a.K, a.V, num_sms);
    while (G > max_cluster) G >>= 1;
    cfg.gridDim = dim3((unsigned)G, (unsigned)a.K, (unsigned)a.B);
    cfg.dynamicSmemBytes = draw_smem_bytes(a.V, G);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_draft_sample(const SampleArgs& a, int ddt, int num_sms, cudaStream_t stream) {
    if (ddt == DT_BF16) return launch_sample_t<DT_BF16>(a, num_sms, stream);
    return launch_sample_t<DT_F32>(a, num_sms, stream);
}

}  // namespace sv
