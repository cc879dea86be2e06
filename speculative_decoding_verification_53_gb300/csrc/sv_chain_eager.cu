// sv_chain_eager.cu -- chain verify for small batches: every position staged at once,
// one cluster exchange for all positions' statistics.
//
// The rule is the one of sv_chain.cu ("[논문 리뷰] Fast Inference from
// Transformers via Speculative Decoding", section 2, Step 3; "Speculative
// Decoding and EAGLE", section "정확성 규칙").  For a small batch the
// position-by-position walk pays one cluster exchange per position, so here one
// cluster per batch row brings its chunks of all K+1 target rows (and of the
// K draft-logit rows) into shared memory at kernel entry, computes every
// position's statistics as the copies land, and combines all of them across the
// cluster in a single exchange.  Every CTA then takes the same left-to-right
// decisions locally, and only the first rejection (or the bonus position) costs
// a second exchange: the inverse-CDF draw.  Rows past the first rejection are
// read for nothing; for a batch small enough to leave most SMs idle that costs
// bandwidth that is otherwise unused.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int EAGER_MAX_POS = 16;  // K + 1 positions at most

struct EagerArgs {
    ChainArgs a;
    int t_bytes;      // bytes of one staged target chunk (16-byte multiple)
    int d_bytes;      // bytes of one staged draft-logit chunk (0 for probabilities)
    int probs_bytes;  // area for the rejected position's draft-probability chunk
};

// Per-CTA partial of one position: target (max, sum), draft (max, sum); a NaN sum
// marks a row that contained NaN.  Greedy rows reuse it as (max, index bits, nan, -).
struct EagerInbox {
    float4 part[EAGER_MAX_POS][MAX_CLUSTER];
    float4 gath[EAGER_MAX_POS][MAX_CLUSTER];  // (target value, draft value, has, -) at x_k
};

// Combine, per position, the n partials held by consecutive groups of `width` lanes
// (width a power of two): max first, then one rescale per partial and a sum.
__device__ __forceinline__ void seg_lse(float& m, float& s, int width, float c) {
    float M = m;
    for (int o = width >> 1; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float v = (m > neg_inf() && s == s) ? s * ex2((m - M) * c) : (s == s ? 0.f : s);
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    m = M;
    s = v;
}

__device__ __forceinline__ void seg_argmax(float& v, int& i, int& nan, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        nan |= __shfl_xor_sync(0xffffffffu, nan, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}


template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT) chain_eager_kernel(const EagerArgs E) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    const ChainArgs& a = E.a;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int K = a.K, P = K + 1, V = a.V;
    uint64_t* tbar = reinterpret_cast<uint64_t*>(dsm);  // [P]
    uint64_t* dbar = tbar + EAGER_MAX_POS;               // [K]
    uint64_t* pbar = dbar + EAGER_MAX_POS;               // the probability area
    unsigned char* tslots = dsm + STAGE_HEADER;
    unsigned char* dslots = tslots + (size_t)P * E.t_bytes;
    unsigned char* probs_area = dslots + (size_t)K * E.d_bytes;
    float* tile_sum = reinterpret_cast<float*>(probs_area + E.probs_bytes);
    __shared__ BlockScratch sc;
    __shared__ EagerInbox inbox;
    __shared__ float4 wpart[EAGER_MAX_POS][NW];
    __shared__ float4 cpart[EAGER_MAX_POS], ggat[EAGER_MAX_POS];
    __shared__ float4 stats[EAGER_MAX_POS];
    __shared__ float2 gval[EAGER_MAX_POS];
    __shared__ int s_tok[EAGER_MAX_POS], s_res[4];
    __shared__ float s_r[EAGER_MAX_POS], s_u[EAGER_MAX_POS], s_qx[EAGER_MAX_POS], s_ap[EAGER_MAX_POS];
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)

    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* tbase = reinterpret_cast<const unsigned char*>(a.target) + (size_t)b * P * V * tsz;
    const unsigned char* dbase = reinterpret_cast<const unsigned char*>(a.draft) + (size_t)b * K * V * dsz;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // 1. every target chunk of the row is requested at once
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * EAGER_MAX_POS + 1; ++i) mbar_init(&tbar[i], 1);
        fence_mbar_init();
        for (int k = 0; k < P; ++k) {
            mbar_arrive_expect_tx(&tbar[k], (uint32_t)n * tsz);
            if (n) bulk_g2s(tslots + (size_t)k * E.t_bytes, tbase + ((size_t)k * V + lo) * tsz, (uint32_t)n * tsz, &tbar[k]);
        }
    }
    const float T = a.temperature ? a.temperature[b] : 0.f;
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool draft_rows = !greedy && DK == DK_LOGITS;
    if (threadIdx.x == 0 && !greedy) {
        if (DK == DK_LOGITS) {
            for (int k = 0; k < K; ++k) {
                mbar_arrive_expect_tx(&dbar[k], (uint32_t)n * dsz);
                if (n)
                    bulk_g2s(dslots + (size_t)k * E.d_bytes, dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz,
                             &dbar[k]);
            }
        } else if (n) {
            for (int k = 0; k < K; ++k) prefetch_l2(dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz);
        }
    }
    int tok_bad = 0;
    if ((int)threadIdx.x < K) {
        const int x = a.tokens[(size_t)b * K + threadIdx.x];
        s_tok[threadIdx.x] = x;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    if (threadIdx.x >= 32 && (int)threadIdx.x < 32 + P) {  // warp 1: the Philox blocks
        const int k = threadIdx.x - 32;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, s_r[k], s_u[k]);
    }
    if (DK == DK_PROBS && !greedy && threadIdx.x >= 64 && (int)threadIdx.x < 64 + K) {  // warp 2: q(x_k)
        const int k = threadIdx.x - 64;
        const int x = a.tokens[(size_t)b * K + k];
        s_qx[k] = (x >= 0 && x < V) ? __ldg(reinterpret_cast<const float*>(dbase) + (size_t)k * V + x) : 0.f;
    }
    const bool tokens_bad = __syncthreads_or(tok_bad) != 0;

    // 2. per-position statistics as the copies land; warp partials into shared memory
    for (int k = 0; k < P; ++k) {
        bool ok = mbar_wait_bounded(&tbar[k], 0);
        if (draft_rows && k < K) ok = mbar_wait_bounded(&dbar[k], 0) && ok;
        const unsigned char* tb = tslots + (size_t)k * E.t_bytes;
        const unsigned char* db = dslots + (size_t)k * E.d_bytes;
        if (greedy) {
            ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
            if (!ok) am.bad = 1;
            argmax_warp_reduce(am);
            if (lane == 0) wpart[k][warp] = make_float4(am.v, __int_as_float(am.i), __int_as_float(am.bad), 0.f);
        } else {
            LSE ts = smem_thread_lse<TDT>(tb, n, c);
            LSE ds{neg_inf(), 0.f, 0};
            if (draft_rows && k < K) ds = smem_thread_lse<DDT>(db, n, c);
            if (!ok) ts.bad = 1;
            if (DK == DK_LOGITS) lse2_warp_reduce(ts, ds, c);
            else lse_warp_reduce(ts, c);
            if (lane == 0)
                wpart[k][warp] = make_float4(ts.m, ts.bad ? __int_as_float(0x7fffffff) : ts.s, ds.m,
                                             ds.bad ? __int_as_float(0x7fffffff) : ds.s);
            if (threadIdx.x == 0) {  // the entries at x_k, when this CTA's chunk holds them
                const int x = (k < K && !tokens_bad) ? s_tok[k] : -1;
                const bool own = x >= lo && x < hi;
                ggat[k] = make_float4(own ? smem_elem<TDT>(tb, x - lo) : 0.f,
                                      (own && draft_rows) ? smem_elem<DDT>(db, x - lo) : 0.f, own ? 1.f : 0.f, 0.f);
            }
        }
    }
    __syncthreads();
    // 3. this CTA's partial of every position (segments of NW lanes), pushed to every peer
    if (warp == 0) {
        constexpr int PER = 32 / NW;  // positions per round
        for (int base = 0; base < P; base += PER) {
            const int k = base + lane / NW, q = lane % NW;
            float4 v = k < P ? wpart[k][q] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
            if (greedy) {
                float mv = v.x;
                int mi = k < P ? __float_as_int(v.y) : 0x7fffffff, nan = k < P ? __float_as_int(v.z) : 0;
                seg_argmax(mv, mi, nan, NW);
                v = make_float4(mv, __int_as_float(mi), __int_as_float(nan), 0.f);
            } else {
                seg_lse(v.x, v.y, NW, c);
                if (DK == DK_LOGITS) seg_lse(v.z, v.w, NW, c);
            }
            if (q == 0 && k < P) cpart[k] = v;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * P; i += NT) {
        const int peer = i % G, k = i / G;
        dsmem_st_v4(dsmem_addr(&inbox.part[k][g], (uint32_t)peer), cpart[k]);
        if (!greedy) dsmem_st_v4(dsmem_addr(&inbox.gath[k][g], (uint32_t)peer), ggat[k]);
    }
    cluster_sync_all();
    // 4. every CTA combines the G partials of every position, identically
    if (warp == 0) {
        int width = 1;
        while (width < G) width <<= 1;
        const int per = 32 / width;
        for (int base = 0; base < P; base += per) {
            const int k = base + lane / width, q = lane % width;
            float4 v = (k < P && q < G) ? inbox.part[k][q] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
            if (greedy) {
                float mv = v.x;
                int mi = (k < P && q < G) ? __float_as_int(v.y) : 0x7fffffff;
                int nan = (k < P && q < G) ? __float_as_int(v.z) : 0;
                seg_argmax(mv, mi, nan, width);
                v = make_float4(mv, __int_as_float(mi), __int_as_float(nan), 0.f);
            } else {
                seg_lse(v.x, v.y, width, c);
                if (DK == DK_LOGITS) seg_lse(v.z, v.w, width, c);
            }
            if (q == 0 && k < P) stats[k] = v;
        }
    }
    if (!greedy && (int)threadIdx.x >= 32 && (int)threadIdx.x < 32 + P) {  // the gathered entries
        const int k = threadIdx.x - 32;
        float2 gv = make_float2(0.f, 0.f);
        for (int q = 0; q < G; ++q) {
            const float4 e = inbox.gath[k][q];
            if (e.z != 0.f) { gv = make_float2(e.x, e.y); break; }
        }
        gval[k] = gv;
    }
    __syncthreads();

    // 5. left-to-right decisions, identical in every CTA (thread 0 decides, all read)
    if (threadIdx.x == 0) {
        int j = -1, inval = tokens_bad ? 1 : 0;
        for (int k = 0; k < P && !inval; ++k) {
            const float4 st = stats[k];
            if (greedy) {
                const int am = __float_as_int(st.y);
                if (__float_as_int(st.z) || !(st.x > neg_inf()) || st.x == pos_inf()) { inval = 1; break; }
                if (k < K && s_tok[k] == am) { s_ap[k] = 1.f; continue; }
                if (k < K) s_ap[k] = 0.f;
                j = k;
                s_res[1] = am;
                break;
            }
            const bool tbad = st.y != st.y || !(st.x > neg_inf()) || st.x == pos_inf();
            const bool dbad = DK == DK_LOGITS && k < K && (st.w != st.w || !(st.z > neg_inf()) || st.z == pos_inf());
            if (tbad || dbad) { inval = 1; break; }
            if (k == K) { j = K; break; }
            const float px = ex2((gval[k].x - st.x) * c) * (1.f / st.y);
            const float qx = (DK == DK_LOGITS) ? ex2((gval[k].y - st.z) * c) * (1.f / st.w) : s_qx[k];
            if (DK == DK_PROBS && (!(qx >= 0.f) || qx == pos_inf())) { inval = 1; break; }
            const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
            s_ap[k] = fminf(ratio, 1.f);
            if (s_r[k] < ratio) continue;
            j = k;
            break;
        }
        s_res[0] = j;
        s_res[2] = inval;
    }
    __syncthreads();
    int j = s_res[0];
    bool invalid = s_res[2] != 0;
    int final_tok = greedy ? s_res[1] : -1, writer = 0;
    int phase = 0;
    // 6. the draw at j (sampling rows): the replacement from the residual, or the bonus
    if (!invalid && !greedy) {
        const float4 st = stats[j];
        const float inv_st = 1.f / st.y;
        const float inv_sd = (DK == DK_LOGITS && j < K) ? 1.f / st.w : 0.f;
        const unsigned char* tb = tslots + (size_t)j * E.t_bytes;
        int dfail = 0;
        const unsigned char* qb = dslots + (size_t)j * E.d_bytes;
        if (DK == DK_PROBS && j < K) {
            if (threadIdx.x == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(pbar, (uint32_t)n * dsz);
                if (n) bulk_g2s(probs_area, dbase + ((size_t)j * V + lo) * dsz, (uint32_t)n * dsz, pbar);
            }
            dfail = __syncthreads_or(!mbar_wait_bounded(pbar, 0));
            qb = probs_area;
        }
        DrawResult d;
        if (j < K) {
            const StagedResidual<TDT, DDT, DK> rw{tb, qb, lo, c, st.x, inv_st, st.z, inv_sd};
            d = cluster_draw(rw, lo, hi, s_u[j], tile_sum, sc, phase, dfail);
            if (!d.failed && d.owner < 0) {  // the residual has no mass: draw from p_j
                const StagedP<TDT> pw{tb, lo, c, st.x, inv_st};
                d = cluster_draw(pw, lo, hi, s_u[j], tile_sum, sc, phase);
            }
        } else {
            const StagedP<TDT> pw{tb, lo, c, st.x, inv_st};
            d = cluster_draw(pw, lo, hi, s_u[K], tile_sum, sc, phase);
        }
        if (d.failed || d.owner < 0) {
            invalid = true;
        } else {
            final_tok = d.token;
            writer = d.owner;
        }
    }
    __syncthreads();
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * P;
        for (int i = threadIdx.x; i < P; i += NT)
            ot[i] = invalid ? -1 : (i < j ? s_tok[i] : (i == j ? final_tok : -1));
        if (a.out_accept_prob)
            for (int i = threadIdx.x; i < K; i += NT)
                a.out_accept_prob[(size_t)b * K + i] = (invalid || i > j) ? -1.f : s_ap[i];
        if (threadIdx.x == 0) a.out_count[b] = invalid ? 0 : j + 1;
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}


size_t eager_smem_bytes(int V, int K, int G, int tsz, int dsz_logits, int probs, int* t_bytes, int* d_bytes,
                        int* p_bytes) {
    const size_t nvec = (size_t)(V + VEC - 1) / VEC, cmax = ((nvec + G - 1) / G) * VEC;
    const size_t tb = (cmax * tsz + 15) & ~(size_t)15;
    const size_t db = dsz_logits ? ((cmax * dsz_logits + 15) & ~(size_t)15) : 0;
    const size_t pb = probs ? ((cmax * 4 + 15) & ~(size_t)15) : 0;
    if (t_bytes) *t_bytes = (int)tb;
    if (d_bytes) *d_bytes = (int)db;
    if (p_bytes) *p_bytes = (int)pb;
    return STAGE_HEADER + (size_t)(K + 1) * tb + (size_t)K * db + pb + draw_smem_bytes(V, G);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_eager_t(const ChainArgs& a, int G, cudaStream_t stream) {
    auto kern = chain_eager_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    if (a.K + 1 > EAGER_MAX_POS) return cudaErrorInvalidClusterSize;
    EagerArgs E;
    E.a = a;
    const size_t smem = eager_smem_bytes(a.V, a.K, G, TDT == DT_BF16 ? 2 : 4, DK == DK_LOGITS ? (DDT == DT_BF16 ? 2 : 4) : 0,
                                         DK == DK_PROBS ? 1 : 0, &E.t_bytes, &E.d_bytes, &E.probs_bytes);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int maxc = 0;  // 0 when the shared memory does not fit: the caller takes another kernel
    const cudaError_t e = cache.max_cluster((const void*)kern, cfg, &maxc);
    if (e != cudaSuccess) return e;
    if (maxc < G) return cudaErrorInvalidClusterSize;
    cfg.gridDim = dim3((unsigned)G, (unsigned)a.B, 1);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, E);
}

cudaError_t launch_chain_eager(const ChainArgs& a, int tdt, int ddt, int dk, int G, cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_chain_eager_t<DT_BF16, DT_F32, DK_PROBS>(a, G, stream);
        return launch_chain_eager_t<DT_F32, DT_F32, DK_PROBS>(a, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_chain_eager_t<DT_BF16, DT_BF16, DK_LOGITS>(a, G, stream);
        return launch_chain_eager_t<DT_BF16, DT_F32, DK_LOGITS>(a, G, stream);
    }
    if (ddt == DT_BF16) return launch_chain_eager_t<DT_F32, DT_BF16, DK_LOGITS>(a, G, stream);
    return launch_chain_eager_t<DT_F32, DT_F32, DK_LOGITS>(a, G, stream);
}

}  // namespace sv
