// sv_tree_staged.cu -- draft-tree verify with node rows staged in shared memory.
//
// The rule is the one of sv_tree.cu ("Progressive Tree Drafting" summary, section
// "검증"; "Speculative Decoding and EAGLE", section "트리 어텐션 검증"): children
// of the current node are tried in index order; greedy rows descend into the
// child whose token is the argmax; sampling rows keep child c with probability
// min(1, p(t_c)/q(t_c)) and, after a rejection, continue with p <- (p - q)+/Z,
// q(t_c) <- 0, q renormalised; with no child kept (or at a leaf) the last token
// is drawn from the current p.
//
// Here each CTA's chunk of the current node's target and draft rows sits in a
// shared-memory slot (bulk copy on an mbarrier), so every sibling-rejection pass
// and the final draw read shared memory, and the children's rows are prefetched
// into spare slots while the current node is decided: the descent finds its
// next rows already on chip.  Rows of nodes that are neither on the walked path
// nor children of it are never read.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

struct TreeHist {
    int n;
    int x[MAX_NODES];
    float zinv[MAX_NODES + 1];
    float qs[MAX_NODES + 1];
    unsigned char applied[MAX_NODES];
};

// w_n(i), q_n(i) of element i after the recorded rejections (see sv_tree.cu).
__device__ __forceinline__ void hist_state(const TreeHist& hs, int i, float p0, float q0, float& w, float& q) {
    w = p0;
    bool tried = false;
    for (int h = 1; h <= hs.n; ++h) {
        const float qprev = tried ? 0.f : q0 * hs.qs[h - 1];
        if (hs.applied[h - 1]) w = fmaxf(w * hs.zinv[h - 1] - qprev, 0.f);
        tried |= (i == hs.x[h - 1]);
    }
    q = tried ? 0.f : q0 * hs.qs[hs.n];
}

// p0 / q0 of 8 staged elements of the current node (row coordinates).
template <int TDT, int DDT, int DK>
struct StagedNode {
    const unsigned char* tb;
    const unsigned char* db;
    int lo;
    float c, mtc, inv_st, mdc, inv_sd;
    __device__ __forceinline__ void load(int e0, int hi, float p0[VEC], float q0[VEC]) const {
        float l[VEC], d[VEC];
        smem_load8<TDT>(tb, e0 - lo, hi - lo, neg_inf(), l);
        smem_load8<DDT>(db, e0 - lo, hi - lo, DK == DK_LOGITS ? neg_inf() : 0.f, d);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            p0[j] = ex2(fmaf(l[j], c, -mtc)) * inv_st;
            q0[j] = (DK == DK_LOGITS) ? ex2(fmaf(d[j], c, -mdc)) * inv_sd : d[j];
        }
    }
};

template <int TDT, int DDT, int DK>
struct StagedNodeDraw {  // the current p of the node, w_n(i)
    StagedNode<TDT, DDT, DK> row;
    const TreeHist* hs;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        if (hs->n == 0) {
            float l[VEC];
            smem_load8<TDT>(row.tb, e0 - row.lo, hi - row.lo, neg_inf(), l);
#pragma unroll
            for (int j = 0; j < VEC; ++j) w[j] = ex2(fmaf(l[j], row.c, -row.mtc)) * row.inv_st;
            return;
        }
        float p0[VEC], q0[VEC];
        row.load(e0, hi, p0, q0);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            float q;
            hist_state(*hs, e0 + j, p0[j], q0[j], w[j], q);
        }
    }
};


constexpr int TREE_GATHER = 64;  // children whose raw values are prefetched at node entry

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT) tree_staged_kernel(const TreeArgs a, const StageLayout L) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsm);  // one mbarrier per slot
    unsigned char* slots = dsm + STAGE_HEADER;
    float* tile_sum = reinterpret_cast<float*>(slots + (size_t)L.nslot * L.slot_bytes);
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_NODES], s_par[MAX_NODES], s_child[MAX_NODES];
    __shared__ float s_r[MAX_NODES], s_u[MAX_NODES + 1];
    __shared__ float s_rt[TREE_GATHER], s_rd[TREE_GATHER];
    __shared__ int s_out[65], s_path[64];
    __shared__ int s_nchild, s_flag;
    __shared__ TreeHist hs;

    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    const int N = a.N, V = a.V, D = a.max_depth;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* tbase = reinterpret_cast<const unsigned char*>(a.target) + (size_t)b * (N + 1) * V * tsz;
    const unsigned char* dbase = reinterpret_cast<const unsigned char*>(a.draft) + (size_t)b * (N + 1) * V * dsz;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // slot bookkeeping, identical in every thread: the row a slot holds (-1 free), copies in flight
    int slot_row[16];
    uint32_t pend = 0, par = 0;
#pragma unroll
    for (int s = 0; s < 16; ++s) slot_row[s] = -1;
    auto issue_t = [&](int row, int s) {  // target chunk; the phase stays open until complete_issue
        if (threadIdx.x == 0) {
            fence_proxy_async();
            mbar_expect_tx(&bars[s], (uint32_t)n * tsz);
            if (n) bulk_g2s(slots + (size_t)s * L.slot_bytes, tbase + ((size_t)row * V + lo) * tsz, (uint32_t)n * tsz,
                            &bars[s]);
        }
    };
    auto complete_issue = [&](int row, int s, bool with_draft) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&bars[s], with_draft ? (uint32_t)n * dsz : 0u);
            if (with_draft && n)
                bulk_g2s(slots + (size_t)s * L.slot_bytes + L.t_bytes, dbase + ((size_t)row * V + lo) * dsz,
                         (uint32_t)n * dsz, &bars[s]);
        }
    };
    auto wait_slot = [&](int s) -> bool {
        const bool ok = mbar_wait_bounded(&bars[s], (par >> s) & 1u);
        par ^= 1u << s;
        pend &= ~(1u << s);
        return ok;
    };

    // the root's rows are requested first
    if (threadIdx.x == 0) {
        for (int s = 0; s < L.nslot; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    issue_t(0, 0);
    slot_row[0] = 0;
    pend = 1u;
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int t = a.node_tokens[(size_t)b * N + i], p = a.parent[(size_t)b * N + i];
        s_tok[i] = t;
        s_par[i] = p;
        if (t < 0 || t >= V || p < -1 || p >= i) bad = 1;
    }
    for (int i = (int)threadIdx.x - 32; i >= 0 && i <= N; i += NT - 32) {  // Philox blocks (warps 1..)
        float r, u;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)i, r, u);
        if (i < N) s_r[i] = r;
        s_u[i] = u;
    }
    const float T = a.temperature[b];
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool with_draft = !greedy;
    complete_issue(0, 0, with_draft);
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

    int phase = 0, emitted = 0, cur = -1, writer = 0, s_cur = 0;
    while (!invalid) {
        const int row = cur + 1;
        if (warp == 0) {  // children of `cur` in increasing index
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
        // raw values of the children's tokens in this node's rows (sampling), fetched while the copy lands
        if (!greedy && (int)threadIdx.x < nchild && threadIdx.x < TREE_GATHER) {
            const int x = s_tok[s_child[threadIdx.x]];
            s_rt[threadIdx.x] = load_one<TDT>(tbase + (size_t)row * V * tsz, x);
            s_rd[threadIdx.x] = load_one<DDT>(dbase + (size_t)row * V * dsz, x);
        }
        // prefetch the children's rows into free slots
        for (int q = 0; q < nchild; ++q) {
            int s = -1;
            for (int t = 0; t < L.nslot; ++t)
                if (slot_row[t] < 0) { s = t; break; }
            if (s < 0) break;
            if (pend & (1u << s)) (void)wait_slot(s);  // a dropped prefetch still in flight
            const int crow = s_child[q] + 1;
            __syncthreads();
            issue_t(crow, s);
            complete_issue(crow, s, with_draft);
            slot_row[s] = crow;
            pend |= 1u << s;
        }
        const int fail = __syncthreads_or((pend & (1u << s_cur)) ? !wait_slot(s_cur) : 0);
        const unsigned char* tb = slots + (size_t)s_cur * L.slot_bytes;
        const unsigned char* db = tb + L.t_bytes;
        int next = -1;
        if (greedy) {
            ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
            if (fail) am.bad = 1;
            am = cluster_argmax(am, sc, phase);
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            for (int q = 0; q < nchild; ++q)
                if (s_tok[s_child[q]] == am.i) { next = s_child[q]; break; }
            if (threadIdx.x == 0) s_out[emitted] = am.i;
            if (next < 0) { ++emitted; writer = 0; break; }
        } else {
            LSE ts = smem_thread_lse<TDT>(tb, n, c);
            LSE ds{neg_inf(), 0.f, 0};
            if (DK == DK_LOGITS && nchild > 0) ds = smem_thread_lse<DDT>(db, n, c);
            if (fail) ts.bad = 1;
            const PosStats ps = cluster_pos_stats<DK == DK_LOGITS>(ts, ds, c, 0.f, 0.f, 0, sc, phase);
            if (row_bad_s(ps.t) || (DK == DK_LOGITS && nchild > 0 && row_bad_s(ps.d))) { invalid = true; break; }
            const float inv_st = 1.f / ps.t.s;
            const float inv_sd = (DK == DK_LOGITS && nchild > 0) ? 1.f / ps.d.s : 0.f;
            const StagedNode<TDT, DDT, DK> node{tb, db, lo, c, ps.t.m * c, inv_st, ps.d.m * c, inv_sd};
            if (threadIdx.x == 0) {
                hs.n = 0;
                hs.zinv[0] = 1.f;
                hs.qs[0] = 1.f;
            }
            __syncthreads();
            for (int q = 0; q < nchild && !invalid; ++q) {
                const int cidx = s_child[q], x = s_tok[cidx];
                const float rt = q < TREE_GATHER ? s_rt[q] : load_one<TDT>(tbase + (size_t)row * V * tsz, x);
                const float rd = q < TREE_GATHER ? s_rd[q] : load_one<DDT>(dbase + (size_t)row * V * dsz, x);
                const float p0x = ex2(fmaf(rt, c, -node.mtc)) * inv_st;
                const float q0x = (DK == DK_LOGITS) ? ex2(fmaf(rd, c, -node.mdc)) * inv_sd : rd;
                if (DK == DK_PROBS && (!(q0x >= 0.f) || q0x == pos_inf())) { invalid = true; break; }
                float wx, qx;
                hist_state(hs, x, p0x, q0x, wx, qx);
                const float px = wx * hs.zinv[hs.n];
                const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
                if (s_r[cidx] < ratio) { next = cidx; break; }
                // rejected: the next residual mass and q normaliser, from the staged chunk
                float2 part = make_float2(0.f, 0.f);
                const int nh = hs.n;
                for (int e0 = lo + (int)threadIdx.x * VEC; e0 < hi; e0 += NT * VEC) {
                    float p0[VEC], q0[VEC];
                    node.load(e0, hi, p0, q0);
#pragma unroll
                    for (int jj = 0; jj < VEC; ++jj) {
                        float w, qq;
                        hist_state(hs, e0 + jj, p0[jj], q0[jj], w, qq);
                        part.x += fmaxf(w * hs.zinv[nh] - qq, 0.f);
                        part.y += (e0 + jj == x) ? 0.f : qq;
                    }
                }
                const float2 tot = cluster_sum2(part, sc, phase);
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
            if (next < 0) {  // no child kept (or a leaf): the last token from the current p
                const StagedNodeDraw<TDT, DDT, DK> dw{node, &hs};
                const DrawResult d = cluster_draw(dw, lo, hi, s_u[row], tile_sum, sc, phase);
                if (threadIdx.x == 0) s_out[emitted] = d.token;
                ++emitted;
                writer = d.owner;
                break;
            }
            if (threadIdx.x == 0) s_out[emitted] = s_tok[next];
        }
        // descend into `next`: its rows are in a slot already, or are requested now
        if (threadIdx.x == 0) s_path[emitted] = next;
        ++emitted;
        cur = next;
        int s_next = -1;
        for (int t = 0; t < L.nslot; ++t)
            if (slot_row[t] == next + 1) s_next = t;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t != s_next) slot_row[t] = -1;
        __syncthreads();  // every read of the previous node's slot is done
        if (s_next < 0) {
            s_next = s_cur;
            if (pend & (1u << s_next)) (void)wait_slot(s_next);
            issue_t(next + 1, s_next);
            complete_issue(next + 1, s_next, with_draft);
            pend |= 1u << s_next;
        }
        slot_row[s_next] = next + 1;
        s_cur = s_next;
    }
    for (int s = 0; s < L.nslot; ++s)  // copies in flight must land before the CTA exits
        if (pend & (1u << s)) (void)wait_slot(s);
    __syncthreads();
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * (D + 1);
        int32_t* op = a.out_path + (size_t)b * D;
        for (int i = threadIdx.x; i <= D; i += NT) ot[i] = (!invalid && i < emitted) ? s_out[i] : -1;
        for (int i = threadIdx.x; i < D; i += NT) op[i] = (!invalid && i < emitted - 1) ? s_path[i] : -1;
        if (threadIdx.x == 0) a.out_count[b] = invalid ? 0 : emitted;
    }
    cluster_sync_all();
}


template <int TDT, int DDT, int DK>
static cudaError_t launch_tree_staged_t(const TreeArgs& a, const StageLayout& L, int G, cudaStream_t stream) {
    auto kern = tree_staged_kernel<TDT, DDT, DK>;
    static int max_dyn = -1;
    if (max_dyn < 0) {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        const int m = optin - (int)fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, m);
        if (e != cudaSuccess) return e;
        max_dyn = m;
    }
    StageLayout Lk = L;
    size_t smem = STAGE_HEADER + (size_t)Lk.nslot * Lk.slot_bytes + draw_smem_bytes(a.V, G);
    while (smem > (size_t)max_dyn && Lk.nslot > 1) {  // fewer prefetch slots when static memory is large
        --Lk.nslot;
        smem -= Lk.slot_bytes;
    }
    if (smem > (size_t)max_dyn) return cudaErrorInvalidClusterSize;  // caller takes the streaming kernel
    static size_t cached_smem = 0;
    static int cached_max = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if (cached_smem != smem) {
        cfg.gridDim = dim3(MAX_CLUSTER, 1, 1);
        int m = 0;
        cudaError_t e = cudaOccupancyMaxPotentialClusterSize(&m, kern, &cfg);
        if (e != cudaSuccess) return e;
        cached_max = m;
        cached_smem = smem;
    }
    if (cached_max < G) return cudaErrorInvalidClusterSize;
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
    return cudaLaunchKernelEx(&cfg, kern, a, Lk);
}

cudaError_t launch_tree_staged(const TreeArgs& a, const StageLayout& L, int tdt, int ddt, int dk, int G,
                               cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_tree_staged_t<DT_BF16, DT_F32, DK_PROBS>(a, L, G, stream);
        return launch_tree_staged_t<DT_F32, DT_F32, DK_PROBS>(a, L, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_tree_staged_t<DT_BF16, DT_BF16, DK_LOGITS>(a, L, G, stream);
        return launch_tree_staged_t<DT_BF16, DT_F32, DK_LOGITS>(a, L, G, stream);
    }
    if (ddt == DT_BF16) return launch_tree_staged_t<DT_F32, DT_BF16, DK_LOGITS>(a, L, G, stream);
    return launch_tree_staged_t<DT_F32, DT_F32, DK_LOGITS>(a, L, G, stream);
}

}  // namespace sv
