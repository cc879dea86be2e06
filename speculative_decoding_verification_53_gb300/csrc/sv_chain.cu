// sv_chain.cu -- chain verify and greedy acceptance, one thread-block cluster per batch row.
//
// The rule ("[논문 리뷰] Fast Inference from Transformers via Speculative Decoding",
// section 2, Step 3; "Speculative Decoding and EAGLE", section "정확성 규칙"):
// positions are checked left to right, x_k is kept with probability
// min(1, p_k(x_k)/q_k(x_k)); the first rejection draws a replacement from
// (p_k - q_k)+ and ends the round; when all K pass, a bonus token is drawn from
// p_K.  Greedy rows keep x_k while it equals argmax p_k and end with that argmax.
//
// Layout of the work: the V entries of a row are split into G contiguous chunks,
// one per CTA of a G-CTA cluster; each CTA streams its chunk with 16-byte loads,
// reduces to (max, sum of exp2) or (max, argmax) and the cluster combines the G
// partials through distributed shared memory in rank order, so every CTA holds
// the same statistics and takes the same decisions.  Only rows up to the first
// rejection are read.  The replacement draw is an inverse-CDF search split the
// same way (sv_common.cuh, cluster_draw).
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

template <int TDT>
struct PWeights {  // w_i = p_i (the bonus draw, or the fallback of an empty residual)
    static constexpr int kTilesInFlight = 4;  // global loads: several in flight per lane
    const void* trow;
    float c, m, inv_s;
    bool al;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC];
        load8<TDT>(trow, e0, hi, al, neg_inf(), l);
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[j] = ex2((l[j] - m) * c) * inv_s;
    }
};

template <int TDT, int DDT, int DK>
struct ResidualWeights {  // w_i = max(0, p_i - q_i)
    static constexpr int kTilesInFlight = 4;  // global loads: several in flight per lane
    const void* trow;
    const void* drow;
    float c, mt, inv_st, md, inv_sd;
    bool at, ad;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC], d[VEC];
        load8<TDT>(trow, e0, hi, at, neg_inf(), l);
        load8<DDT>(drow, e0, hi, ad, DK == DK_LOGITS ? neg_inf() : 0.f, d);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float p = ex2((l[j] - mt) * c) * inv_st;
            const float q = (DK == DK_LOGITS) ? ex2((d[j] - md) * c) * inv_sd : d[j];
            w[j] = fmaxf(p - q, 0.f);
        }
    }
};

__device__ __forceinline__ bool row_bad(const LSE& s) {
    return s.bad || !(s.m > neg_inf()) || s.m == pos_inf();
}

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT) chain_kernel(const ChainArgs a) {
    extern __shared__ float tile_sum[];
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_K];
    __shared__ float s_r[MAX_K + 1], s_u[MAX_K + 1], s_ap[MAX_K];
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)

    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    const int K = a.K, V = a.V;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const float T = a.temperature ? a.temperature[b] : 0.f;
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const size_t tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;

    int tok_bad = 0;
    for (int k = threadIdx.x; k < K; k += NT) {
        const int x = a.tokens[(size_t)b * K + k];
        s_tok[k] = x;
        s_ap[k] = -1.f;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    if (!greedy)
        for (int k = threadIdx.x; k <= K; k += NT) slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, s_r[k], s_u[k]);
    bool invalid = __syncthreads_or(tok_bad) != 0;

    // tmo: some wait of the row gave up (this CTA's, or a peer's flag seen in an exchange)
    int phase = 0, j = -1, final_tok = -1, writer = 0, tmo = 0;
    for (int k = 0; k <= K && !invalid; ++k) {
        const void* trow = (const char*)a.target + ((size_t)b * (K + 1) + k) * (size_t)V * tsz;
        const bool at = ((uintptr_t)trow & 15) == 0;
        if (greedy) {
            ArgMax am = thread_argmax<TDT>(trow, lo, hi, at);
            am = cluster_argmax(am, sc, phase);
            if (am.bad & BAD_TIMEOUT) tmo = 1;
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            if (k < K && s_tok[k] == am.i) {
                if (threadIdx.x == 0) s_ap[k] = 1.f;
                continue;
            }
            if (k < K && threadIdx.x == 0) s_ap[k] = 0.f;
            j = k;
            final_tok = am.i;
            writer = 0;
            break;
        }
        const void* drow = (k < K) ? (const char*)a.draft + ((size_t)b * K + k) * (size_t)V * dsz : nullptr;
        const bool ad = ((uintptr_t)drow & 15) == 0;
        LSE ts = thread_lse<TDT>(trow, lo, hi, at, c);
        LSE ds{neg_inf(), 0.f, 0};
        if (DK == DK_LOGITS && k < K) ds = thread_lse<DDT>(drow, lo, hi, ad, c);
        cluster_lse2(ts, ds, c, sc, phase);
        if ((ts.bad | ds.bad) & BAD_TIMEOUT) tmo = 1;
        if (row_bad(ts) || (DK == DK_LOGITS && k < K && row_bad(ds))) { invalid = true; break; }
        const float inv_st = 1.f / ts.s;
        if (k == K) {  // every draft accepted: bonus token from p_K
            const PWeights<TDT> pw{trow, c, ts.m, inv_st, at};
            const DrawResult d = cluster_draw(pw, lo, hi, s_u[K], tile_sum, sc, phase);
            if (d.failed) { tmo = 1; invalid = true; break; }
            j = K;
            final_tok = d.token;
            writer = d.owner;
            break;
        }
        const int x = s_tok[k];
        const float px = ex2((load_one<TDT>(trow, x) - ts.m) * c) * inv_st;
        float qx, inv_sd = 0.f;
        if (DK == DK_LOGITS) {
            inv_sd = 1.f / ds.s;
            qx = ex2((load_one<DDT>(drow, x) - ds.m) * c) * inv_sd;
        } else {
            qx = load_one<DT_F32>(drow, x);
            if (!(qx >= 0.f) || qx == pos_inf()) { invalid = true; break; }
        }
        const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
        if (threadIdx.x == 0) s_ap[k] = fminf(ratio, 1.f);
        if (s_r[k] < ratio) continue;
        // first rejection: replacement from the residual (p_k - q_k)+
        const ResidualWeights<TDT, DDT, DK> rw{trow, drow, c, ts.m, inv_st, ds.m, inv_sd, at, ad};
        DrawResult d = cluster_draw(rw, lo, hi, s_u[k], tile_sum, sc, phase);
        if (d.failed) { tmo = 1; invalid = true; break; }
        if (d.owner < 0) {  // the residual has no mass: draw from p_k
            const PWeights<TDT> pw{trow, c, ts.m, inv_st, at};
            d = cluster_draw(pw, lo, hi, s_u[k], tile_sum, sc, phase);
            if (d.failed) { tmo = 1; invalid = true; break; }
        }
        j = k;
        final_tok = d.token;
        writer = d.owner;
        break;
    }
    __syncthreads();
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * (K + 1);
        for (int i = threadIdx.x; i <= K; i += NT)
            ot[i] = invalid ? -1 : (i < j ? s_tok[i] : (i == j ? final_tok : -1));
        if (a.out_accept_prob)
            for (int i = threadIdx.x; i < K; i += NT) a.out_accept_prob[(size_t)b * K + i] = invalid ? -1.f : s_ap[i];
        if (threadIdx.x == 0) a.out_count[b] = invalid ? (tmo ? SV_COUNT_TIMEOUT : 0) : j + 1;
    }
    // Leave together: when every exchange completes, the walk is the same in every CTA of
    // the cluster and nothing is pushed into a CTA after its last exchange; but a CTA
    // whose bounded wait gave up may have left the walk early while a peer still pushes
    // into its inbox.  Every wait before this barrier is bounded, so every CTA reaches
    // it.  A CTA that saw a timeout then marks the row (after any other writer).
    cluster_sync_all();
    if (tmo && threadIdx.x == 0) a.out_count[b] = SV_COUNT_TIMEOUT;
}

size_t draw_smem_bytes(int V, int cluster) {
    const long long nvec = (V + VEC - 1) / VEC;
    const long long chunk = ((nvec + cluster - 1) / cluster + 1) * VEC;
    return (size_t)((chunk + TILE - 1) / TILE + 1) * sizeof(float);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_t(const ChainArgs& a, int G, cudaStream_t stream) {
    auto kern = chain_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    const cudaError_t e = cache.pick_cluster((const void*)kern, cfg, G, [&](int g) { return draw_smem_bytes(a.V, g); }, &G);
    if (e != cudaSuccess) return e;
    if (G == 0) return cudaErrorInvalidValue;  // no cluster size fits the draw's tile sums
    cfg.gridDim = dim3((unsigned)G, (unsigned)a.B, 1);
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

cudaError_t launch_chain(const ChainArgs& a, int tdt, int ddt, int dk, int G, cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_chain_t<DT_BF16, DT_F32, DK_PROBS>(a, G, stream);
        return launch_chain_t<DT_F32, DT_F32, DK_PROBS>(a, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_chain_t<DT_BF16, DT_BF16, DK_LOGITS>(a, G, stream);
        return launch_chain_t<DT_BF16, DT_F32, DK_LOGITS>(a, G, stream);
    }
    if (ddt == DT_BF16) return launch_chain_t<DT_F32, DT_BF16, DK_LOGITS>(a, G, stream);
    return launch_chain_t<DT_F32, DT_F32, DK_LOGITS>(a, G, stream);
}

}  // namespace sv
