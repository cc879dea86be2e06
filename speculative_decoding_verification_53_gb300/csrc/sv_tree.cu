// sv_tree.cu -- draft-tree verify, one thread-block cluster per batch row.
//
// The rule ("Progressive Tree Drafting" summary, section "검증": greedy tree
// acceptance and sampling acceptance without replacement from normalised
// probabilities; "Speculative Decoding and EAGLE", section "트리 어텐션 검증":
// the longest accepted branch): starting at the root, the children of the
// current node are tried in increasing node index.  Greedy rows descend into the
// child whose token is the argmax of the current row.  Sampling rows keep child
// c with probability min(1, p(t_c)/q(t_c)); after a rejection
// p <- (p - q)+ / |(p - q)+|_1 (kept when that mass is zero), q(t_c) <- 0 and q is
// renormalised; when no child is kept (or at a leaf) the last token is drawn
// from the current p.
//
// After h rejections at a node the current distributions are functions of the
// node's original p0, q0 and a short history (tried tokens, residual masses, q
// normalisers), so each element is recomputed from the row on demand: one pass
// over the row per rejection (for the next residual mass and q normaliser) and
// one inverse-CDF pass for the final draw.  Rows of nodes off the walked path
// are never read.
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

// Rejection history at the current node, kept in shared memory.
struct TreeHistory {
    int n;                     // rejections so far (h = 1..n)
    int x[MAX_NODES];          // tried token of step h (index h-1)
    float zinv[MAX_NODES + 1]; // 1/Z of the residual after h steps (index h); zinv[0] = 1
    float qs[MAX_NODES + 1];   // q normaliser after h steps (index h); qs[0] = 1
    unsigned char applied[MAX_NODES];  // step h replaced p by the residual (mass > 0)
};

// Current (unnormalised) weight w_n(i) of element i and its q_n(i), from p0(i), q0(i).
__device__ __forceinline__ void tree_state_at(const TreeHistory& hs, int i, float p0, float q0, float& w,
                                              float& q) {
    w = p0;
    bool tried = false;
    for (int h = 1; h <= hs.n; ++h) {
        const float qprev = tried ? 0.f : q0 * hs.qs[h - 1];
        if (hs.applied[h - 1]) w = fmaxf(w * hs.zinv[h - 1] - qprev, 0.f);
        tried |= (i == hs.x[h - 1]);
    }
    q = tried ? 0.f : q0 * hs.qs[hs.n];
}

template <int TDT, int DDT, int DK>
struct TreeRow {
    const void* trow;
    const void* drow;
    float c, mt, inv_st, md, inv_sd;
    bool at, ad;
    __device__ __forceinline__ void load(int e0, int hi, float p0[VEC], float q0[VEC]) const {
        float l[VEC], d[VEC];
        load8<TDT>(trow, e0, hi, at, neg_inf(), l);
        load8<DDT>(drow, e0, hi, ad, DK == DK_LOGITS ? neg_inf() : 0.f, d);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            p0[j] = ex2((l[j] - mt) * c) * inv_st;
            q0[j] = (DK == DK_LOGITS) ? ex2((d[j] - md) * c) * inv_sd : d[j];
        }
    }
};

// Draw weights: the current p of the node, w_n(i).
template <int TDT, int DDT, int DK>
struct TreeDrawWeights {
    TreeRow<TDT, DDT, DK> row;
    const TreeHistory* hs;
    bool has_q;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        if (!has_q) {  // no rejection happened: plain p0, no draft row needed
            float l[VEC];
            load8<TDT>(row.trow, e0, hi, row.at, neg_inf(), l);
#pragma unroll
            for (int j = 0; j < VEC; ++j) w[j] = ex2((l[j] - row.mt) * row.c) * row.inv_st;
            return;
        }
        float p0[VEC], q0[VEC];
        row.load(e0, hi, p0, q0);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            float q;
            tree_state_at(*hs, e0 + j, p0[j], q0[j], w[j], q);
        }
    }
};

__device__ __forceinline__ bool tree_row_bad(const LSE& s) {
    return s.bad || !(s.m > neg_inf()) || s.m == pos_inf();
}

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT) tree_kernel(const TreeArgs a) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    extern __shared__ float tile_sum[];
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_NODES], s_par[MAX_NODES], s_child[MAX_NODES];
    __shared__ float s_r[MAX_NODES];
    __shared__ int s_out[65], s_path[64];
    __shared__ int s_nchild, s_flag;
    __shared__ TreeHistory hs;
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)

    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    const int N = a.N, V = a.V, D = a.max_depth;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const float T = a.temperature[b];
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const size_t tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int t = a.node_tokens[(size_t)b * N + i], p = a.parent[(size_t)b * N + i];
        s_tok[i] = t;
        s_par[i] = p;
        if (t < 0 || t >= V || p < -1 || p >= i) bad = 1;
    }
    if (!greedy)
        for (int i = threadIdx.x; i < N; i += NT) {
            float r, u;
            slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)i, r, u);
            s_r[i] = r;
        }
    bool invalid = __syncthreads_or(bad) != 0;
    if (!invalid && threadIdx.x == 0) {  // every node's depth must fit max_depth
        int deep = 0;
        for (int i = 0; i < N; ++i) {
            const int p = s_par[i];
            const int d = p < 0 ? 1 : s_child[p] + 1;  // s_child doubles as depth scratch here
            s_child[i] = d;
            if (d > D) deep = 1;
        }
        s_flag = deep;
    }
    __syncthreads();
    if (!invalid) invalid = s_flag != 0;
    __syncthreads();

    // tmo: some wait of the row gave up (this CTA's, or a peer's flag seen in an exchange)
    int phase = 0, emitted = 0, cur = -1, writer = 0, tmo = 0;
    while (!invalid) {
        const int row = cur + 1;
        const void* trow = (const char*)a.target + ((size_t)b * (N + 1) + row) * (size_t)V * tsz;
        const bool at = ((uintptr_t)trow & 15) == 0;
        // children of `cur` in increasing index (warp 0, ballot compaction)
        if (warp == 0) {
            int cnt = 0;
            for (int base = 0; base < N; base += 32) {
                const int i = base + lane;
                const bool is_child = i < N && s_par[i] == cur;
                const unsigned m = __ballot_sync(0xffffffffu, is_child);
                if (is_child) s_child[cnt + __popc(m & ((1u << lane) - 1u))] = i;
                cnt += __popc(m);
            }
            if (lane == 0) s_nchild = cnt;
        }
        __syncthreads();
        const int nchild = s_nchild;
        if (greedy) {
            ArgMax am = thread_argmax<TDT>(trow, lo, hi, at);
            am = cluster_argmax(am, sc, phase);
            if (am.bad & BAD_TIMEOUT) tmo = 1;
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            int next = -1;
            for (int q = 0; q < nchild; ++q)
                if (s_tok[s_child[q]] == am.i) { next = s_child[q]; break; }
            if (threadIdx.x == 0) s_out[emitted] = am.i;
            if (next < 0) { ++emitted; writer = 0; break; }
            if (threadIdx.x == 0) s_path[emitted] = next;
            ++emitted;
            cur = next;
            __syncthreads();
            continue;
        }
        const void* drow = (const char*)a.draft + ((size_t)b * (N + 1) + row) * (size_t)V * dsz;
        const bool ad = ((uintptr_t)drow & 15) == 0;
        LSE ts = thread_lse<TDT>(trow, lo, hi, at, c);
        LSE ds{neg_inf(), 0.f, 0};
        if (DK == DK_LOGITS && nchild > 0) ds = thread_lse<DDT>(drow, lo, hi, ad, c);
        cluster_lse2(ts, ds, c, sc, phase);
        if ((ts.bad | ds.bad) & BAD_TIMEOUT) tmo = 1;
        if (tree_row_bad(ts) || (DK == DK_LOGITS && nchild > 0 && tree_row_bad(ds))) { invalid = true; break; }
        const TreeRow<TDT, DDT, DK> rw{trow, drow, c, ts.m, 1.f / ts.s, ds.m, DK == DK_LOGITS ? 1.f / ds.s : 0.f,
                                       at, ad};
        if (threadIdx.x == 0) {
            hs.n = 0;
            hs.zinv[0] = 1.f;
            hs.qs[0] = 1.f;
        }
        __syncthreads();
        int next = -1;
        for (int q = 0; q < nchild && !invalid; ++q) {
            const int cidx = s_child[q], x = s_tok[cidx];
            float p0x = ex2((load_one<TDT>(trow, x) - rw.mt) * c) * rw.inv_st;
            float q0x = (DK == DK_LOGITS) ? ex2((load_one<DDT>(drow, x) - rw.md) * c) * rw.inv_sd
                                          : load_one<DT_F32>(drow, x);
            if (DK == DK_PROBS && (!(q0x >= 0.f) || q0x == pos_inf())) { invalid = true; break; }
            float wx, qx;
            tree_state_at(hs, x, p0x, q0x, wx, qx);
            const float px = wx * hs.zinv[hs.n];
            const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
            if (s_r[cidx] < ratio) { next = cidx; break; }
            // rejected: next residual mass and q normaliser over the whole row
            float2 part = make_float2(0.f, 0.f);
            const int nh = hs.n;
            for (int e0 = lo + (int)threadIdx.x * VEC; e0 < hi; e0 += NT * VEC) {
                float p0[VEC], q0[VEC];
                rw.load(e0, hi, p0, q0);
#pragma unroll
                for (int jj = 0; jj < VEC; ++jj) {
                    float w, qq;
                    tree_state_at(hs, e0 + jj, p0[jj], q0[jj], w, qq);
                    part.x += fmaxf(w * hs.zinv[nh] - qq, 0.f);
                    part.y += (e0 + jj == x) ? 0.f : qq;
                }
            }
            const float2 tot = cluster_sum2(part, sc, phase);
            if (tot.x != tot.x) {  // the exchange gave up (NaN sums)
                tmo = 1;
                invalid = true;
                break;
            }
            if (threadIdx.x == 0) {
                // without replacement the tried token leaves q and q is renormalised;
                // i.i.d. siblings leave q as it is (no token recorded, no rescale)
                const bool iid = a.sibling_rule == SV_SIBLINGS_IID;
                hs.x[nh] = iid ? -1 : x;
                hs.applied[nh] = tot.x > 0.f ? 1 : 0;
                hs.zinv[nh + 1] = tot.x > 0.f ? 1.f / tot.x : hs.zinv[nh];
                hs.qs[nh + 1] = (!iid && tot.y > 0.f) ? hs.qs[nh] / tot.y : hs.qs[nh];
                hs.n = nh + 1;
            }
            __syncthreads();
        }
        if (invalid) break;
        if (next >= 0) {
            if (threadIdx.x == 0) {
                s_out[emitted] = s_tok[next];
                s_path[emitted] = next;
            }
            ++emitted;
            cur = next;
            __syncthreads();
            continue;
        }
        float r_unused, u;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)row, r_unused, u);
        const TreeDrawWeights<TDT, DDT, DK> dw{rw, &hs, hs.n > 0};
        const DrawResult d = cluster_draw(dw, lo, hi, u, tile_sum, sc, phase);
        if (d.failed || d.owner < 0) {
            tmo = d.failed ? 1 : tmo;
            invalid = true;
            break;
        }
        if (threadIdx.x == 0) s_out[emitted] = d.token;
        ++emitted;
        writer = d.owner;
        break;
    }
    __syncthreads();
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * (D + 1);
        int32_t* op = a.out_path + (size_t)b * D;
        for (int i = threadIdx.x; i <= D; i += NT) ot[i] = (!invalid && i < emitted) ? s_out[i] : -1;
        for (int i = threadIdx.x; i < D; i += NT) op[i] = (!invalid && i < emitted - 1) ? s_path[i] : -1;
        if (threadIdx.x == 0) a.out_count[b] = invalid ? (tmo ? SV_COUNT_TIMEOUT : 0) : emitted;
    }
    // Leave together: when every exchange completes, the walk is the same in every CTA of
    // the cluster and nothing is pushed into a CTA after its last exchange; but a CTA
    // whose bounded wait gave up may have left the walk early while a peer still pushes
    // into its inbox.  Every wait before this barrier is bounded, so every CTA reaches
    // it.  A CTA that saw a timeout then marks the row (after any other writer).
    cluster_sync_all();
    if (tmo && threadIdx.x == 0) a.out_count[b] = SV_COUNT_TIMEOUT;
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_tree_t(const TreeArgs& a, int G, cudaStream_t stream) {
    auto kern = tree_kernel<TDT, DDT, DK>;
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

cudaError_t launch_tree(const TreeArgs& a, int tdt, int ddt, int dk, int G, cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_tree_t<DT_BF16, DT_F32, DK_PROBS>(a, G, stream);
        return launch_tree_t<DT_F32, DT_F32, DK_PROBS>(a, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_tree_t<DT_BF16, DT_BF16, DK_LOGITS>(a, G, stream);
        return launch_tree_t<DT_BF16, DT_F32, DK_LOGITS>(a, G, stream);
    }
    if (ddt == DT_BF16) return launch_tree_t<DT_F32, DT_BF16, DK_LOGITS>(a, G, stream);
    return launch_tree_t<DT_F32, DT_F32, DK_LOGITS>(a, G, stream);
}

}  // namespace sv
