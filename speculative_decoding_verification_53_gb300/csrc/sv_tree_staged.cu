// sv_tree_staged.cu -- draft-tree verify with node rows staged in shared memory.
//
// The rule is the one of sv_tree.cu ("Progressive Tree Drafting" summary, section
// "검증"; "Speculative Decoding and EAGLE", section "트리 어텐션 검증"): children
// of the current node are tried in index order; greedy rows descend into the
// child whose token is the argmax; sampling rows keep child c with probability
// min(1, p(t_c)/q(t_c)) and, after a rejection, continue with p <- (p - q)+/Z,
// q(t_c) <- 0, q renormalised (i.i.d. siblings: q left as it is); with no child
// kept (or at a leaf) the last token is drawn from the current p.
//
// Each CTA's chunk of the current node's target and draft rows sits in a
// shared-memory slot (bulk copy on an mbarrier), and the children's rows are
// prefetched into spare slots while the current node is decided.  The current
// (unnormalised) weights w_h after h rejections are kept in an fp32 array of the
// chunk and updated in place by each rejection pass, w_{h+1} = (w_h / Z_h - q_h)+,
// so a pass and the final draw cost O(1) per element whatever the number of
// rejections; the tokens tried so far are a bitmask of the chunk.  The acceptance
// test of a child evaluates the same recursion for its one token from the
// recorded history (the same operations in the same order, so both agree bit for
// bit).  Rows of nodes that are neither on the walked path nor children of it
// are never read.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

// Rejection history at the current node (views into shared memory).
struct TreeHist {
    int* x;          // token tried at step h (-1: none recorded, i.i.d. siblings)
    float* zinv;     // 1/Z after h steps (index h); zinv[0] = 1
    float* qs;       // q scale after h steps (index h); qs[0] = 1
    int* applied;    // step h replaced p by the residual (its mass was > 0)
};

// w_n(i), q_n(i) of element i after n recorded rejections, from p0(i), q0(i).
__device__ __forceinline__ void hist_state(const TreeHist& hs, int n, int i, float p0, float q0, float& w, float& q) {
    w = p0;
    bool tried = false;
    for (int h = 1; h <= n; ++h) {
        const float qprev = tried ? 0.f : q0 * hs.qs[h - 1];
        if (hs.applied[h - 1]) w = fmaxf(fmaf(w, hs.zinv[h - 1], -qprev), 0.f);  // as the rejection pass
        tried |= (i == hs.x[h - 1]);
    }
    q = tried ? 0.f : q0 * hs.qs[n];
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

// The current p of the node for the draw: the kept weights after a rejection, else p0.
template <int TDT>
struct StagedNodeP {
    const unsigned char* tb;
    const float* wbuf;
    int lo;
    float c, mtc, inv_st;
    bool mat;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        if (mat) {
            smem_load8<DT_F32>(reinterpret_cast<const unsigned char*>(wbuf), e0 - lo, hi - lo, 0.f, w);
            return;
        }
        float l[VEC];
        smem_load8<TDT>(tb, e0 - lo, hi - lo, neg_inf(), l);
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[j] = ex2(fmaf(l[j], c, -mtc)) * inv_st;
    }
};

constexpr int TREE_GATHER = 64;  // children whose raw values are prefetched at node entry

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT, 2) tree_staged_kernel(const TreeArgs a, const StageLayout L) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ BlockScratch sc;
    __shared__ float s_rt[TREE_GATHER], s_rd[TREE_GATHER];
    __shared__ int s_out[65], s_path[64];
    __shared__ int s_nchild, s_hn;
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)

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

    // dynamic shared memory: barriers | per-tree arrays | slots | weights, tried mask | tile sums
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsm);  // one mbarrier per slot
    int* s_tok = reinterpret_cast<int*>(dsm + STAGE_HEADER);
    int* s_par = s_tok + N;
    int* s_child = s_par + N;  // depth counts first, then the children of the current node
    int* s_jump = s_child + N;
    float* s_r = reinterpret_cast<float*>(s_jump + N);
    float* s_u = s_r + N;  // N + 1
    int* h_x = reinterpret_cast<int*>(s_u + N + 1);
    float* h_zinv = reinterpret_cast<float*>(h_x + N);  // N + 1
    float* h_qs = h_zinv + N + 1;                         // N + 1
    int* h_applied = reinterpret_cast<int*>(h_qs + N + 1);
    const TreeHist hs{h_x, h_zinv, h_qs, h_applied};
    unsigned char* slots = dsm + STAGE_HEADER + tree_array_bytes(N);
    const int cap = chunk_cap(V, G);
    float* wbuf = reinterpret_cast<float*>(slots + (size_t)L.nslot * L.slot_bytes);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(wbuf) +
                                                  (((size_t)cap * 4 + 15) & ~(size_t)15));
    float* tile_sum = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(wbuf) + tree_work_bytes(V, G));

    // barriers and the Philox blocks (kernel parameters only) before the dependency wait
    if (threadIdx.x == 0) {
        for (int s = 0; s < L.nslot; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    for (int i = (int)threadIdx.x - 32; i >= 0 && i <= N; i += NT - 32) {  // warps 1..
        float r, u;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)i, r, u);
        if (i < N) s_r[i] = r;
        s_u[i] = u;
    }
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this

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
    auto issue_t_nofence = [&](int row, int s) {  // issue_t after the caller's proxy fence
        if (threadIdx.x == 0) {
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
    // thread 0 polls; every call is followed by a CTA barrier that releases the others
    auto wait_slot = [&](int s) -> bool {
        const bool ok = threadIdx.x != 0 || mbar_wait_bounded(&bars[s], (par >> s) & 1u);
        par ^= 1u << s;
        pend &= ~(1u << s);
        return ok;
    };

    // the root's rows are requested first
    issue_t(0, 0);
    slot_row[0] = 0;
    pend = 1u;
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int t = a.node_tokens[(size_t)b * N + i], p = a.parent[(size_t)b * N + i];
        s_tok[i] = t;
        s_par[i] = p;
        s_child[i] = 1;
        s_jump[i] = p;
        if (t < 0 || t >= V || p < -1 || p >= i) bad = 1;
    }
    const float T = a.temperature[b];
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool with_draft = !greedy;
    complete_issue(0, 0, with_draft);
    bool invalid = __syncthreads_or(bad) != 0;
    int tmo = 0;  // some wait of the row gave up (this CTA's, or a peer's flag seen in an exchange)
    int drain_fail = 0;  // a wait for a copy that was not used gave up (this thread)
    if (!invalid) {
        // every node's depth must fit max_depth: depths by pointer jumping on (count, target)
        // pairs, read / barrier / write rounds; a node stops at the root or beyond D
        constexpr int PER = MAX_NODES / NT;
        int dcur[PER], jcur[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int i = (int)threadIdx.x + q * NT;
            dcur[q] = 1;
            jcur[q] = i < N ? s_par[i] : -1;
        }
        auto live = [&](int q) { return jcur[q] >= 0 && dcur[q] <= D; };
        for (;;) {
            int any = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) any |= live(q) ? 1 : 0;
            if (!__syncthreads_or(any)) break;
            int dd[PER], jj[PER];
            bool act[PER];
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                act[q] = live(q);
                dd[q] = act[q] ? s_child[jcur[q]] : 0;
                jj[q] = act[q] ? s_jump[jcur[q]] : -1;
            }
            __syncthreads();
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                if (!act[q]) continue;
                const int i = (int)threadIdx.x + q * NT;
                dcur[q] += dd[q];
                jcur[q] = jj[q];
                s_child[i] = dcur[q];
                s_jump[i] = jcur[q];
            }
        }
        int deep = 0;
#pragma unroll
        for (int q = 0; q < PER; ++q) deep |= dcur[q] > D ? 1 : 0;
        invalid = __syncthreads_or(deep) != 0;
    }

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
        // prefetch the children's rows into free slots (before the gathers below: the proxy
        // fence of a copy would otherwise wait for thread 0's outstanding loads).  A free
        // slot's reads ended at the barrier the walk passed when it descended; a dropped
        // prefetch still in flight is waited for first (by thread 0, which issues every
        // copy).  Then one barrier and one proxy fence cover the whole batch of copies.
        {
            int sq[16], nq = 0;
            for (int q = 0; q < nchild && nq < 16; ++q) {
                int s = -1;
                for (int t = 0; t < L.nslot; ++t)
                    if (slot_row[t] < 0) { s = t; break; }
                if (s < 0) break;
                if (pend & (1u << s)) drain_fail |= wait_slot(s) ? 0 : 1;  // a dropped prefetch still in flight
                slot_row[s] = s_child[q] + 1;
                pend |= 1u << s;
                sq[nq++] = s;
            }
            if (nq > 0) {
                __syncthreads();
                if (threadIdx.x == 0) fence_proxy_async();
                for (int i = 0; i < nq; ++i) {
                    issue_t_nofence(slot_row[sq[i]], sq[i]);
                    complete_issue(slot_row[sq[i]], sq[i], with_draft);
                }
            }
        }
        // raw values of the children's tokens in this node's rows (sampling): the loads are
        // issued now and their values stored after the statistics, so the latency overlaps
        const bool gat = !greedy && (int)threadIdx.x < nchild && threadIdx.x < TREE_GATHER;
        float g_rt = 0.f, g_rd = 0.f;
        if (gat) {
            const int x = s_tok[s_child[threadIdx.x]];
            g_rt = load_one<TDT>(tbase + (size_t)row * V * tsz, x);
            g_rd = load_one<DDT>(dbase + (size_t)row * V * dsz, x);
        }
        const int fail = __syncthreads_or((pend & (1u << s_cur)) ? !wait_slot(s_cur) : 0);
        const unsigned char* tb = slots + (size_t)s_cur * L.slot_bytes;
        const unsigned char* db = tb + L.t_bytes;
        int next = -1;
        if (greedy) {
            ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
            if (fail) am.bad |= BAD_TIMEOUT;
            am = cluster_argmax(am, sc, phase);
            if (am.bad & BAD_TIMEOUT) tmo = 1;
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            for (int q = 0; q < nchild; ++q)
                if (s_tok[s_child[q]] == am.i) { next = s_child[q]; break; }
            if (threadIdx.x == 0) s_out[emitted] = am.i;
            if (next < 0) { ++emitted; writer = 0; break; }
        } else {
            LSE ts, ds{neg_inf(), 0.f, 0};
            if (DK == DK_LOGITS && nchild > 0) {
                smem_thread_lse2<TDT, DDT>(tb, db, n, c, ts, ds);
            } else {
                ts = smem_thread_lse<TDT>(tb, n, c);
            }
            if (fail) ts.bad |= BAD_TIMEOUT;
            if (gat) {
                s_rt[threadIdx.x] = g_rt;
                s_rd[threadIdx.x] = g_rd;
            }
            for (int w = threadIdx.x; w < (cap + 31) / 32; w += NT) tmask[w] = 0u;  // nothing tried yet
            if (threadIdx.x == 0) {
                s_hn = 0;
                h_zinv[0] = 1.f;
                h_qs[0] = 1.f;
            }
            // (the combine's barriers publish the gathered values, the mask and the history)
            const PosStats ps = cluster_pos_stats<DK == DK_LOGITS>(ts, ds, c, 0.f, 0.f, 0, sc, phase);
            if ((ps.t.bad | ps.d.bad) & BAD_TIMEOUT) tmo = 1;
            if (row_bad_s(ps.t) || (DK == DK_LOGITS && nchild > 0 && row_bad_s(ps.d))) { invalid = true; break; }
            const float inv_st = 1.f / ps.t.s;
            const float inv_sd = (DK == DK_LOGITS && nchild > 0) ? 1.f / ps.d.s : 0.f;
            const StagedNode<TDT, DDT, DK> node{tb, db, lo, c, ps.t.m * c, inv_st, ps.d.m * c, inv_sd};
            const bool iid = a.sibling_rule == SV_SIBLINGS_IID;
            bool wmat = false;  // wbuf holds w_h (else the current weights are still p0)
            for (int q = 0; q < nchild && !invalid; ++q) {
                const int cidx = s_child[q], x = s_tok[cidx];
                const float rt = q < TREE_GATHER ? s_rt[q] : load_one<TDT>(tbase + (size_t)row * V * tsz, x);
                const float rd = q < TREE_GATHER ? s_rd[q] : load_one<DDT>(dbase + (size_t)row * V * dsz, x);
                const float p0x = ex2(fmaf(rt, c, -node.mtc)) * inv_st;
                const float q0x = (DK == DK_LOGITS) ? ex2(fmaf(rd, c, -node.mdc)) * inv_sd : rd;
                if (DK == DK_PROBS && (!(q0x >= 0.f) || q0x == pos_inf())) { invalid = true; break; }
                const int nh = s_hn;
                float wx, qx;
                hist_state(hs, nh, x, p0x, q0x, wx, qx);
                const float px = wx * h_zinv[nh];
                const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
                if (s_r[cidx] < ratio) { next = cidx; break; }
                // rejected: w_{h+1} = (w_h / Z_h - q_h)+ in place, with the residual mass and
                // the mass of q without x
                const float zi = h_zinv[nh], qsn = h_qs[nh];
                // the arithmetic of hist_state, two lanes at a time: q0 = 2^(d c - md c) / S_d,
                // w' = max(fma(w, 1/Z, -q0 qs), 0) (the negated q scale gives -q0 qs exactly)
                const float2 cc = make_float2(c, c), zi2 = make_float2(zi, zi), nqs = make_float2(-qsn, -qsn);
                const float2 md2 = make_float2(-node.mdc, -node.mdc), isd = make_float2(inv_sd, inv_sd);
                const float2 mt2 = make_float2(-node.mtc, -node.mtc), ist = make_float2(inv_st, inv_st);
                float2 part = make_float2(0.f, 0.f);
                for (int e0 = lo + (int)threadIdx.x * VEC; e0 < hi; e0 += NT * VEC) {
                    const int o = e0 - lo;
                    float wv[VEC], d[VEC];
                    smem_load8<DDT>(db, o, n, DK == DK_LOGITS ? neg_inf() : 0.f, d);
                    if (wmat) {
                        smem_load8<DT_F32>(reinterpret_cast<const unsigned char*>(wbuf), o, n, 0.f, wv);
                    } else {
                        float l[VEC];
                        smem_load8<TDT>(tb, o, n, neg_inf(), l);
#pragma unroll
                        for (int j = 0; j < VEC; j += 2) {
                            const float2 y = ffma2(make_float2(l[j], l[j + 1]), cc, mt2);
                            const float2 p = fmul2(make_float2(ex2(y.x), ex2(y.y)), ist);
                            wv[j] = p.x;
                            wv[j + 1] = p.y;
                        }
                    }
                    const uint32_t tw = (tmask[o >> 5] >> (o & 31)) & 0xffu;  // 8 elements share a mask word
                    float r[VEC], nq[VEC];
#pragma unroll
                    for (int j = 0; j < VEC; j += 2) {
                        float2 q0 = make_float2(d[j], d[j + 1]);
                        if (DK == DK_LOGITS) {
                            const float2 y = ffma2(q0, cc, md2);
                            q0 = fmul2(make_float2(ex2(y.x), ex2(y.y)), isd);
                        }
                        const float2 nq2 = fmul2(q0, nqs);
                        nq[j] = nq2.x;
                        nq[j + 1] = nq2.y;
                    }
                    if (tw) {  // tried tokens in this vector weigh nothing in q
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            if ((tw >> j) & 1u) nq[j] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < VEC; j += 2) {
                        const float2 rr = ffma2(make_float2(wv[j], wv[j + 1]), zi2, make_float2(nq[j], nq[j + 1]));
                        r[j] = fmaxf(rr.x, 0.f);
                        r[j + 1] = fmaxf(rr.y, 0.f);
                    }
                    part.x += sum8(r);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) part.y -= (e0 + j == x) ? 0.f : nq[j];
                    if (o + VEC <= n) {
                        *reinterpret_cast<float4*>(wbuf + o) = make_float4(r[0], r[1], r[2], r[3]);
                        *reinterpret_cast<float4*>(wbuf + o + 4) = make_float4(r[4], r[5], r[6], r[7]);
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            if (o + j < n) wbuf[o + j] = r[j];
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
                    h_x[nh] = iid ? -1 : x;
                    h_applied[nh] = tot.x > 0.f ? 1 : 0;
                    h_zinv[nh + 1] = tot.x > 0.f ? 1.f / tot.x : zi;
                    h_qs[nh + 1] = (!iid && tot.y > 0.f) ? qsn / tot.y : qsn;
                    s_hn = nh + 1;
                    if (!iid && x >= lo && x < hi) tmask[(x - lo) >> 5] |= 1u << ((x - lo) & 31);
                }
                __syncthreads();
                if (tot.x > 0.f) {
                    wmat = true;
                } else if (wmat) {
                    // the residual had no mass, so w stays w_h, which the pass overwrote:
                    // rebuild it from the history (the pages' rule keeps p in this case)
                    for (int e0 = lo + (int)threadIdx.x * VEC; e0 < hi; e0 += NT * VEC) {
                        float p0[VEC], q0[VEC];
                        node.load(e0, hi, p0, q0);
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            float w, qq;
                            hist_state(hs, nh + 1, e0 + j, p0[j], q0[j], w, qq);
                            if (e0 + j < hi) wbuf[e0 - lo + j] = w;
                        }
                    }
                    __syncthreads();
                }
            }
            if (invalid) break;
            if (next < 0) {  // no child kept (or a leaf): the last token from the current p
                const StagedNodeP<TDT> pw{tb, wbuf, lo, c, node.mtc, inv_st, wmat};
                const DrawResult d = cluster_draw(pw, lo, hi, s_u[row], tile_sum, sc, phase);
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
            if (pend & (1u << s_next)) drain_fail |= wait_slot(s_next) ? 0 : 1;
            issue_t(next + 1, s_next);
            complete_issue(next + 1, s_next, with_draft);
            pend |= 1u << s_next;
        }
        slot_row[s_next] = next + 1;
        s_cur = s_next;
    }
    for (int s = 0; s < L.nslot; ++s)  // copies in flight must land before the CTA exits
        if (pend & (1u << s)) drain_fail |= wait_slot(s) ? 0 : 1;
    // a wait for a copy that was not used (a dropped prefetch) that gave up: the slot may
    // still have been written after it was reused, so the row reports a timeout
    if (__syncthreads_or(drain_fail)) tmo = 1;
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
static cudaError_t launch_tree_staged_t(const TreeArgs& a, const StageLayout& L, int G, cudaStream_t stream) {
    auto kern = tree_staged_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    int max_dyn = 0;
    {
        const cudaError_t e = cache.setup((const void*)kern, &max_dyn);
        if (e != cudaSuccess) return e;
    }
    StageLayout Lk = L;
    size_t smem = STAGE_HEADER + tree_array_bytes(a.N) + (size_t)Lk.nslot * Lk.slot_bytes + tree_work_bytes(a.V, G) +
                  draw_smem_bytes(a.V, G);
    while (smem > (size_t)max_dyn && Lk.nslot > 1) {  // fewer prefetch slots when static memory is large
        --Lk.nslot;
        smem -= Lk.slot_bytes;
    }
    if (smem > (size_t)max_dyn) return cudaErrorInvalidClusterSize;  // caller takes the streaming kernel
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int maxc = 0;
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
