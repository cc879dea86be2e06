// sv_chain_staged.cu -- chain verify with each CTA's row chunks staged in shared memory.
//
// Same rule and the same cluster split as sv_chain.cu ("[논문 리뷰] Fast Inference
// from Transformers via Speculative Decoding", section 2, Step 3; "Speculative
// Decoding and EAGLE", section "정확성 규칙"), but the CTA's chunk of the target
// row (and of the draft-logit row) of position k is brought into shared memory
// by a bulk copy, so the statistics, the gathered entries at x_k and the
// replacement draw all read shared memory: every row crosses HBM once.  A ring
// of `nslot` slots lets a small batch prefetch the next positions while the
// current one is decided; a large batch uses one slot (no speculative reads) and
// relies on the other CTAs of the SM to hide latency.  Draft probabilities are
// only needed at the rejected position: that chunk is copied on demand (after an
// optional L2 prefetch at kernel start).
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT, 4) chain_staged_kernel(const ChainArgs a, const StageLayout L) {
    extern __shared__ __align__(128) unsigned char dsm[];
    // mbarriers: [0, nslot) target chunks, [nslot, 2 nslot) draft-logit chunks, [2 nslot] probabilities
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsm);
    uint64_t* tbar = bars;
    uint64_t* dbar = bars + L.nslot;
    uint64_t* pbar = bars + 2 * L.nslot;
    unsigned char* slots = dsm + STAGE_HEADER;
    unsigned char* probs_area = slots + (size_t)L.nslot * L.slot_bytes;
    float* tile_sum = reinterpret_cast<float*>(probs_area + L.probs_bytes);
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_K];
    __shared__ float s_r[MAX_K + 1], s_u[MAX_K + 1], s_ap[MAX_K];
    __shared__ float s_qx;
    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    const int K = a.K, V = a.V;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* tbase = reinterpret_cast<const unsigned char*>(a.target) + (size_t)b * (K + 1) * V * tsz;
    const unsigned char* dbase = reinterpret_cast<const unsigned char*>(a.draft) + (size_t)b * K * V * dsz;
    const int first = (K + 1 < L.nslot) ? K + 1 : L.nslot;  // positions staged up front

    // Test hook (off unless stall_row is set): this row's first target copy is announced
    // on its barrier but never issued, so the bounded wait for it runs out (after
    // stall_ns) and the row reports a timeout; no copy is in flight for it.
    const bool stall = b == a.stall_row;
    const uint32_t wait_ns = stall ? a.stall_ns : WAIT_LIMIT_NS;
    auto issue_t = [&](int k) {
        const int s = k % L.nslot;
        fence_proxy_async();
        mbar_arrive_expect_tx(&tbar[s], (uint32_t)n * tsz);
        if (n && !(stall && k == 0))
            bulk_g2s(slots + (size_t)s * L.slot_bytes, tbase + ((size_t)k * V + lo) * tsz, (uint32_t)n * tsz, &tbar[s]);
    };
    auto issue_d = [&](int k) {
        const int s = k % L.nslot;
        mbar_arrive_expect_tx(&dbar[s], (uint32_t)n * dsz);
        if (n)
            bulk_g2s(slots + (size_t)s * L.slot_bytes + L.t_bytes, dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz,
                     &dbar[s]);
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i <= 2 * L.nslot; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    // the Philox blocks (kernel parameters only) on warps 1.., before the dependency wait
    // and off warp 0's path to the first copies; greedy rows simply never use them
    for (int k = (int)threadIdx.x - 32; k >= 0 && k <= K; k += NT - 32)
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, s_r[k], s_u[k]);
    // inbox barriers of the cluster exchanges: set up and arrive now (no global memory
    // is touched), wait in xchg_ready() just before the first exchange
    xchg_init_arrive(sc);
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    // Start-up, shortest path to the first chunks first: the temperature and the tokens
    // are requested ahead of the bulk copies (so they do not queue behind them), the
    // target chunks go out at once, the draft-logit chunks as soon as the temperature
    // says the row samples.  The wait at the cluster barrier that makes every CTA's
    // exchange barriers exist and the token checks overlap the copies.
    const float T = a.temperature ? a.temperature[b] : 0.f;
    static_assert(NT >= MAX_K, "one drafted token per thread");
    const int tok_reg = (int)threadIdx.x < K ? a.tokens[(size_t)b * K + threadIdx.x] : 0;
    if (threadIdx.x == 0)
        for (int k = 0; k < first; ++k) issue_t(k);
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool draft_rows = !greedy && DK == DK_LOGITS;  // draft-logit rows take part in the statistics
    // they travel with the target rows through the slots, or (d_direct: large batches, whose
    // slots then hold twice as many rows on chip) are streamed from global memory
    const bool d_direct = DK == DK_LOGITS && L.d_direct != 0;
    const bool copy_d = draft_rows && !d_direct;
    if (threadIdx.x == 0) {
        if (copy_d)
            for (int k = 0; k < first && k < K; ++k) issue_d(k);
        if (d_direct && draft_rows && K > 0 && n) prefetch_l2(dbase + (size_t)lo * dsz, (uint32_t)n * dsz);
        if (DK == DK_PROBS && !greedy && L.prefetch_l2 && n)
            for (int k = 0; k < K; ++k) prefetch_l2(dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz);
    }
    uint32_t tpar = 0, dpar = 0, tpend = 0, dpend = 0;  // per-slot phase parity / copy-in-flight bits
    for (int k = 0; k < first; ++k) {
        tpend |= 1u << k;
        if (copy_d && k < K) dpend |= 1u << k;
    }

    int tok_bad = 0;
    if ((int)threadIdx.x < K) {
        s_tok[threadIdx.x] = tok_reg;
        s_ap[threadIdx.x] = -1.f;
        if (tok_reg < 0 || tok_reg >= V) tok_bad = 1;
    }
    bool invalid = __syncthreads_or(tok_bad) != 0;
    xchg_ready();

    auto issue = [&](int k) {  // refill: position k into slot k % nslot (its previous reads are done)
        const int s = k % L.nslot;
        if (threadIdx.x == 0) {
            issue_t(k);
            if (copy_d && k < K) issue_d(k);
            // a draft-logit row streamed directly is announced to L2 now: its statistics then
            // stream from L2 while the target chunk lands (no extra bytes: the row is read anyway)
            if (d_direct && draft_rows && k < K && n) prefetch_l2(dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz);
        }
        tpend |= 1u << s;
        if (copy_d && k < K) dpend |= 1u << s;
    };
    // Both chunks of slot s (the draft one only if requested).  Thread 0 polls the
    // barriers; every call is followed by a CTA barrier, which carries its observation of
    // the landed copies to the other threads (they wait there without taking issue slots).
    auto wait_slot = [&](int s) -> bool {
        bool ok = true;
        if (tpend & (1u << s)) {
            if (threadIdx.x == 0) ok = mbar_wait_bounded_ns(&tbar[s], (tpar >> s) & 1u, wait_ns);
            tpar ^= 1u << s;
            tpend &= ~(1u << s);
        }
        if (dpend & (1u << s)) {
            if (threadIdx.x == 0) ok = mbar_wait_bounded(&dbar[s], (dpar >> s) & 1u) && ok;
            dpar ^= 1u << s;
            dpend &= ~(1u << s);
        }
        return ok;
    };
    int next_issue = first;

    // tmo: some wait of the row gave up (this CTA's, or a peer's flag seen in an exchange)
    int phase = 0, j = -1, final_tok = -1, writer = 0, tmo = 0;
    for (int k = 0; k <= K && !invalid; ++k) {
        const int s = k % L.nslot;
        const int x = k < K ? s_tok[k] : -1;
        float qx_load = 0.f;  // q(x_k) for draft probabilities, loaded while the copy lands
        if (DK == DK_PROBS && !greedy && k < K && threadIdx.x == 0)
            qx_load = __ldg(reinterpret_cast<const float*>(dbase) + (size_t)k * V + x);
        // a draft-logit row read directly is reduced while the target chunk lands
        const unsigned char* drow = dbase + (size_t)k * V * dsz;
        LSE ds_direct{neg_inf(), 0.f, 0};
        if (d_direct && draft_rows && k < K) ds_direct = global_thread_lse<DDT>(drow, lo, hi, c);
        const int fail = __syncthreads_or(!wait_slot(s));
        if (DK == DK_PROBS && !greedy && k < K && threadIdx.x == 0) s_qx = qx_load;
        const unsigned char* tb = slots + (size_t)s * L.slot_bytes;
        const unsigned char* db = tb + L.t_bytes;
        if (greedy) {
            ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
            if (fail) am.bad |= BAD_TIMEOUT;
            am = cluster_argmax(am, sc, phase);
            if (am.bad & BAD_TIMEOUT) tmo = 1;
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            if (k < K && x == am.i) {
                if (threadIdx.x == 0) s_ap[k] = 1.f;
                if (next_issue <= K) issue(next_issue++);
                continue;
            }
            if (k < K && threadIdx.x == 0) s_ap[k] = 0.f;
            j = k;
            final_tok = am.i;
            writer = 0;
            break;
        }
        LSE ts, ds{neg_inf(), 0.f, 0};
        if (draft_rows && k < K && !d_direct) {
            smem_thread_lse2<TDT, DDT>(tb, db, n, c, ts, ds);
        } else {
            ts = smem_thread_lse<TDT>(tb, n, c);
            if (draft_rows && k < K) ds = ds_direct;
        }
        if (fail) ts.bad |= BAD_TIMEOUT;
        float tx = 0.f, dx = 0.f;
        int has = 0;
        if (threadIdx.x == 0 && x >= lo && x < hi) {
            tx = smem_elem<TDT>(tb, x - lo);
            if (draft_rows) dx = d_direct ? load_one<DDT>(drow, x) : smem_elem<DDT>(db, x - lo);
            has = 1;
        }
        const PosStats ps = cluster_pos_stats<DK == DK_LOGITS>(ts, ds, c, tx, dx, has, sc, phase);
        if ((ps.t.bad | ps.d.bad) & BAD_TIMEOUT) tmo = 1;
        if (row_bad_s(ps.t) || (draft_rows && k < K && row_bad_s(ps.d))) { invalid = true; break; }
        const float inv_st = 1.f / ps.t.s;
        if (k == K) {  // every draft accepted: bonus token from p_K
            const StagedP<TDT> pw{tb, lo, c, ps.t.m, inv_st};
            const DrawResult d = cluster_draw(pw, lo, hi, s_u[K], tile_sum, sc, phase);
            if (d.failed) { tmo = 1; invalid = true; break; }
            j = K;
            final_tok = d.token;
            writer = d.owner;
            break;
        }
        const float px = ex2((ps.tx - ps.t.m) * c) * inv_st;
        float qx, inv_sd = 0.f;
        if (DK == DK_LOGITS) {
            inv_sd = 1.f / ps.d.s;
            qx = ex2((ps.dx - ps.d.m) * c) * inv_sd;
        } else {
            qx = s_qx;
            if (!(qx >= 0.f) || qx == pos_inf()) { invalid = true; break; }
        }
        const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
        if (threadIdx.x == 0) s_ap[k] = fminf(ratio, 1.f);
        if (s_r[k] < ratio) {
            if (next_issue <= K) issue(next_issue++);
            continue;
        }
        // first rejection: replacement from the residual (p_k - q_k)+
        int dfail = 0;
        const unsigned char* qb = db;
        if (DK == DK_PROBS) {
            if (threadIdx.x == 0 && n) {
                fence_proxy_async();
                mbar_arrive_expect_tx(pbar, (uint32_t)n * dsz);
                bulk_g2s(probs_area, dbase + ((size_t)k * V + lo) * dsz, (uint32_t)n * dsz, pbar);
            } else if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(pbar, 0u);
            }
            dfail = __syncthreads_or(threadIdx.x == 0 && !mbar_wait_bounded(pbar, 0u));
            qb = probs_area;
        }
        DrawResult d;
        if (d_direct) {
            const StagedResidualD<TDT, DDT> rw{tb, drow, lo, c, ps.t.m, ps.d.m, ps.t.s / ps.d.s};
            d = cluster_draw(rw, lo, hi, s_u[k], tile_sum, sc, phase, dfail);
        } else {
            const StagedResidual<TDT, DDT, DK> rw{tb, qb, lo, c, ps.t.m, inv_st, ps.d.m, inv_sd};
            d = cluster_draw(rw, lo, hi, s_u[k], tile_sum, sc, phase, dfail);
        }
        if (d.failed) { tmo = 1; invalid = true; break; }
        if (d.owner < 0) {  // the residual has no mass: draw from p_k
            const StagedP<TDT> pw{tb, lo, c, ps.t.m, inv_st};
            d = cluster_draw(pw, lo, hi, s_u[k], tile_sum, sc, phase);
            if (d.failed) { tmo = 1; invalid = true; break; }
        }
        j = k;
        final_tok = d.token;
        writer = d.owner;
        break;
    }
    // copies still in flight (prefetched positions never reached) must land before the CTA
    // exits; a wait that gives up here reports the row as timed out
    int drain_fail = 0;
    for (int s = 0; s < L.nslot; ++s)
        if ((tpend | dpend) & (1u << s)) drain_fail |= wait_slot(s) ? 0 : 1;
    if (__syncthreads_or(drain_fail)) tmo = 1;
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * (K + 1);
        for (int i = threadIdx.x; i <= K; i += NT)
            ot[i] = invalid ? -1 : (i < j ? s_tok[i] : (i == j ? final_tok : -1));
        if (a.out_accept_prob)
            for (int i = threadIdx.x; i < K; i += NT)
                a.out_accept_prob[(size_t)b * K + i] = invalid ? -1.f : s_ap[i];
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

size_t staged_smem_bytes(const StageLayout& L, int V, int G) {
    return STAGE_HEADER + (size_t)L.nslot * L.slot_bytes + L.probs_bytes + draw_smem_bytes(V, G);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_staged_t(const ChainArgs& a, const StageLayout& L, int G, cudaStream_t stream) {
    auto kern = chain_staged_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    const size_t smem = staged_smem_bytes(L, a.V, G);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    cfg.dynamicSmemBytes = smem;
    int maxc = 0;  // largest co-scheduled cluster; 0 when the shared memory does not fit
    const cudaError_t e = cache.max_cluster((const void*)kern, cfg, &maxc);
    if (e != cudaSuccess) return e;
    if (maxc < G) return cudaErrorInvalidClusterSize;  // caller picks another shape or kernel
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
    return cudaLaunchKernelEx(&cfg, kern, a, L);
}

cudaError_t launch_chain_staged(const ChainArgs& a, const StageLayout& L, int tdt, int ddt, int dk, int G,
                                cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_chain_staged_t<DT_BF16, DT_F32, DK_PROBS>(a, L, G, stream);
        return launch_chain_staged_t<DT_F32, DT_F32, DK_PROBS>(a, L, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_chain_staged_t<DT_BF16, DT_BF16, DK_LOGITS>(a, L, G, stream);
        return launch_chain_staged_t<DT_BF16, DT_F32, DK_LOGITS>(a, L, G, stream);
    }
    if (ddt == DT_BF16) return launch_chain_staged_t<DT_F32, DT_BF16, DK_LOGITS>(a, L, G, stream);
    return launch_chain_staged_t<DT_F32, DT_F32, DK_LOGITS>(a, L, G, stream);
}

}  // namespace sv
