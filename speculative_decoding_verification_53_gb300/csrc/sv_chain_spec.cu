// sv_chain_spec.cu -- position-parallel chain verify for small batches.
//
// The rule is the one of sv_chain.cu ("[논문 리뷰] Fast Inference from
// Transformers via Speculative Decoding", section 2, Step 3; "Speculative
// Decoding and EAGLE", section "정확성 규칙"), evaluated in another order.  For a
// small batch the left-to-right walk over positions is latency-bound (one
// cluster exchange per position), so here every position k of every batch row b
// gets its own cluster of G CTAs at once:
//   1. the cluster stages its chunk of target row k (and draft row k), computes
//      the softmax statistics and the acceptance test of x_k (greedy: the argmax);
//   2. if x_k is rejected (or k = K), it completes the draw at k as if k were the
//      first rejection (the replacement from (p_k - q_k)+, or from p_k when that
//      residual is empty; the bonus token from p_K at k = K), inside the cluster
//      and from shared memory;
//   3. one CTA of the cluster writes output slot k (x_k when accepted, else the
//      drawn token) and counts the position in with one 64-bit atomic that also
//      carries the position's reject and invalid bits.
// The last position to arrive for batch row b (no CTA ever waits for another) reads
// the first rejection j and the invalid bits off the value its own atomic
// returned, clears the slots after j and writes the count.  The results are
// those of the left-to-right rule; the price of the shorter critical path is that
// positions past the first rejection are read (and their draws made) for nothing.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

// atomicAdd with acquire-release semantics at GPU scope: this thread's earlier global
// writes are visible to whoever later reads the word's new value, and the writes of
// every earlier adder are visible to this thread afterwards.
__device__ __forceinline__ unsigned long long atomic_add_acq_rel(unsigned long long* p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

// The per-row word in the workspace: arrivals in bits [0, 11), reject bits of
// positions 0..25 in [11, 37), invalid bits of positions 0..25 in [37, 63).  One CTA
// of each position's cluster adds 1 plus the position's two bits, each at most once,
// so the fields never carry into each other.
constexpr int SPEC_COUNT_BITS = 11;
constexpr int SPEC_REJ_SHIFT = 11;
constexpr int SPEC_BAD_SHIFT = 37;
constexpr unsigned long long SPEC_FIELD_MASK = (1ull << SPEC_MAX_POS) - 1ull;

struct SpecWsLayout {
    size_t counter_off, total;
};

__host__ __device__ inline size_t spec_align(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline SpecWsLayout spec_ws_layout(int B, int K) {
    (void)K;
    SpecWsLayout L;
    L.counter_off = 0;
    L.total = spec_align((size_t)B * sizeof(unsigned long long));
    return L;
}

struct SpecArgs {
    ChainArgs a;
    unsigned char* ws;
    SpecWsLayout wl;
    int t_bytes;  // shared-memory offset of the draft chunk
    int d_bytes;  // bytes reserved for the draft chunk (tile sums follow)
};

// Finishing step for batch row b, run by the last CTA to arrive; `word` is the row's
// final counter word (every position's bits are in it).
__device__ __forceinline__ void spec_finish(const SpecArgs& A, int b, bool tok_bad, unsigned long long word) {
    const ChainArgs& a = A.a;
    const int K = a.K;
    const unsigned long long rej = (word >> SPEC_REJ_SHIFT) & SPEC_FIELD_MASK;
    const unsigned long long bad = (word >> SPEC_BAD_SHIFT) & SPEC_FIELD_MASK;
    const int j = rej ? __ffsll((long long)rej) - 1 : K;  // first rejection, or K (every draft kept)
    const bool invalid = tok_bad || (bad & ((2ull << j) - 1ull)) != 0ull;  // rows read up to j must be valid
    int32_t* ot = a.out_tokens + (size_t)b * (K + 1);
    for (int i = threadIdx.x; i <= K; i += NT)
        if (invalid || i > j) ot[i] = -1;
    if (a.out_accept_prob)
        for (int i = threadIdx.x; i < K; i += NT)
            if (invalid || i > j) a.out_accept_prob[(size_t)b * K + i] = -1.f;
    if (threadIdx.x == 0) {
        a.out_count[b] = invalid ? 0 : j + 1;
        *(reinterpret_cast<unsigned long long*>(A.ws + A.wl.counter_off) + b) = 0ull;  // ready for the next call
    }
}


template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT, 1) chain_spec_kernel(const SpecArgs A) {
    const ChainArgs& a = A.a;
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t* tbar = reinterpret_cast<uint64_t*>(dsm);
    uint64_t* dbar = tbar + 1;
    unsigned char* tb = dsm + STAGE_HEADER;                    // target chunk of row (b, k)
    unsigned char* db = tb + A.t_bytes;                        // draft chunk (logits or probabilities)
    float* tile_sum = reinterpret_cast<float*>(db + A.d_bytes);  // the draw's tile sums
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_K];
    __shared__ float s_flt[4];
    __shared__ unsigned long long s_word;  // the row's counter word after this CTA's atomic
    __shared__ int s_last;
    xchg_init(sc);  // inbox barriers of the cluster exchanges (shared memory only)

    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int k = blockIdx.y, b = blockIdx.z;
    const int K = a.K, V = a.V;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* trow = reinterpret_cast<const unsigned char*>(a.target) + ((size_t)b * (K + 1) + k) * V * tsz;
    const unsigned char* drow =
        k < K ? reinterpret_cast<const unsigned char*>(a.draft) + ((size_t)b * K + k) * V * dsz : nullptr;

    // 1. both chunks are requested at once (the draft chunk is wasted on a greedy row,
    // which this small-batch kernel accepts); the temperature, the tokens and the Philox
    // block are fetched and computed meanwhile, independently of each other
    const bool has_draft_row = k < K && a.draft != nullptr;
    if (threadIdx.x == 32) {  // warp 1: the Philox block of slot k (unused on greedy rows)
        float r, u;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, r, u);
        s_flt[0] = r;
        s_flt[1] = u;
    }
    if (threadIdx.x == 0) {
        mbar_init(tbar, 1);
        mbar_init(dbar, 1);
        fence_mbar_init();
    }
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    // The draft chunk goes out with the target chunk when the statistics need it (draft
    // logits); draft probabilities are needed by the draw alone, so their chunk is copied
    // once the target chunk has landed and does not share the SM's copy bandwidth with it.
    auto issue_draft = [&]() {
        mbar_arrive_expect_tx(dbar, (uint32_t)n * dsz);
        if (n) bulk_g2s(db, drow + (size_t)lo * dsz, (uint32_t)n * dsz, dbar);
    };
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(tbar, (uint32_t)n * tsz);
        if (n) bulk_g2s(tb, trow + (size_t)lo * tsz, (uint32_t)n * tsz, tbar);
        if (has_draft_row && DK == DK_LOGITS) issue_draft();
    }
    // draft probabilities: only q(x_k) takes part in the statistics, so thread 0 fetches
    // it directly and the q chunk (needed by the draw alone) keeps landing meanwhile
    float qx_direct = 0.f;
    if (DK == DK_PROBS && threadIdx.x == 0 && has_draft_row) {
        const int xk = a.tokens[(size_t)b * K + k];
        if (xk >= lo && xk < hi) qx_direct = load_one<DT_F32>(drow, xk);
    }
    int tok_bad = 0;
    for (int i = threadIdx.x; i < K; i += NT) {
        const int x = a.tokens[(size_t)b * K + i];
        s_tok[i] = x;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    const float T = a.temperature ? a.temperature[b] : 0.f;
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool tokens_bad = __syncthreads_or(tok_bad) != 0;

    // 2. statistics of row k, the acceptance test of x_k
    // thread 0 polls the copy barriers; the CTA barrier below releases the other threads
    bool ok = threadIdx.x != 0 || mbar_wait_bounded(tbar, 0);
    // (a greedy row never draws: its probability chunk is not copied at all)
    const bool probs_copied = has_draft_row && DK == DK_PROBS && !greedy;
    if (probs_copied && threadIdx.x == 0) issue_draft();
    bool draft_landed = !has_draft_row || (DK == DK_PROBS && !probs_copied);
    if (has_draft_row && DK == DK_LOGITS) {  // draft logits feed the statistics
        ok = (threadIdx.x != 0 || mbar_wait_bounded(dbar, 0)) && ok;
        draft_landed = true;
    }
    const int fail = __syncthreads_or(!ok);
    const int x = (k < K && !tokens_bad) ? s_tok[k] : -1;
    int32_t* slot = a.out_tokens + (size_t)b * (K + 1) + k;  // this position's output slot
    int phase = 0, amax = -1, owner = -1, token = -1;
    bool accept = false, bad = false;
    float ratio = 0.f;
    if (greedy) {
        ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
        if (fail) am.bad |= BAD_TIMEOUT;
        am = cluster_argmax(am, sc, phase);
        bad = am.bad || !(am.v > neg_inf()) || am.v == pos_inf();
        accept = k < K && x == am.i;
        amax = am.i;
    } else {
        LSE ts, ds{neg_inf(), 0.f, 0};
        if (DK == DK_LOGITS && k < K) {
            smem_thread_lse2<TDT, DDT>(tb, db, n, c, ts, ds);
        } else {
            ts = smem_thread_lse<TDT>(tb, n, c);
        }
        if (fail) ts.bad |= BAD_TIMEOUT;
        float tx = 0.f, dx = 0.f;
        int has = 0;
        if (threadIdx.x == 0 && x >= lo && x < hi) {
            tx = smem_elem<TDT>(tb, x - lo);
            dx = (DK == DK_LOGITS) ? smem_elem<DDT>(db, x - lo) : qx_direct;
            has = 1;
        }
        const PosStats ps = cluster_pos_stats<DK == DK_LOGITS>(ts, ds, c, tx, dx, has, sc, phase);
        bad = row_bad_s(ps.t) || (DK == DK_LOGITS && k < K && row_bad_s(ps.d));
        const float inv_st = 1.f / ps.t.s;
        const float inv_sd = (DK == DK_LOGITS && k < K) ? 1.f / ps.d.s : 0.f;
        if (k < K && !bad) {
            const float px = ex2((ps.tx - ps.t.m) * c) * inv_st;
            const float qx = (DK == DK_LOGITS) ? ex2((ps.dx - ps.d.m) * c) * inv_sd : ps.dx;
            if (DK == DK_PROBS && (!(qx >= 0.f) || qx == pos_inf())) bad = true;
            ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
            accept = s_flt[0] < ratio;
        }
        // 3. the draw at k, as if k were the first rejection (the bonus draw at k = K);
        // a kept draft can never be the first rejection, so it needs no draw
        if (!bad && !tokens_bad && !accept) {
            const float u = s_flt[1];
            DrawResult d;
            if (k < K) {
                int dfail = 0;
                if (!draft_landed) {  // the q chunk, for the residual
                    dfail = __syncthreads_or(threadIdx.x == 0 && !mbar_wait_bounded(dbar, 0));
                    draft_landed = true;
                }
                // one CTA per SM here: four tiles in flight per warp shorten the draw's
                // dependent chains (the exp2 pipe has room)
                const InFlight<StagedResidual<TDT, DDT, DK>, 4> rw{{tb, db, lo, c, ps.t.m, inv_st, ps.d.m, inv_sd}};
                d = cluster_draw(rw, lo, hi, u, tile_sum, sc, phase, dfail);
                if (!d.failed && d.owner < 0) {  // the residual has no mass: draw from p_k
                    const InFlight<StagedP<TDT>, 4> pw{{tb, lo, c, ps.t.m, inv_st}};
                    d = cluster_draw(pw, lo, hi, u, tile_sum, sc, phase);
                }
            } else {
                const InFlight<StagedP<TDT>, 4> pw{{tb, lo, c, ps.t.m, inv_st}};
                d = cluster_draw(pw, lo, hi, u, tile_sum, sc, phase);
            }
            if (d.failed || d.owner < 0) bad = true;
            owner = d.owner;
            token = d.token;  // valid in the owner CTA
        }
    }
    // a copy still in flight must land before the CTA exits (a greedy or invalid row
    // never waited for its q chunk); if that bounded wait gives up, the reporting CTA
    // marks the position invalid (another CTA's failed drain is not seen by the reporter)
    int drain_bad = 0;
    if (!draft_landed && threadIdx.x == 0) drain_bad = mbar_wait_bounded(dbar, 0) ? 0 : 1;
    // 4. one CTA reports the position (all of them know its outcome): the owner of the
    // drawn token when there is a draw, else rank 0.  It writes output slot k (the kept
    // draft, the greedy row's argmax or the drawn token) and the acceptance probability,
    // then counts the position in with its reject and invalid bits.
    const bool drawn = !greedy && !bad && !tokens_bad && !accept;
    const int reporter = drawn ? owner : 0;
    if (g == reporter && threadIdx.x == 0) {
        if (!bad && !tokens_bad) {
            *slot = accept ? x : (greedy ? amax : token);
            if (k < K && a.out_accept_prob)
                a.out_accept_prob[(size_t)b * K + k] = greedy ? (accept ? 1.f : 0.f) : fminf(ratio, 1.f);
        }
        unsigned long long inc = 1ull;
        if (k < K && !accept) inc |= 1ull << (SPEC_REJ_SHIFT + k);
        if (bad || drain_bad) inc |= 1ull << (SPEC_BAD_SHIFT + k);
        unsigned long long* word = reinterpret_cast<unsigned long long*>(A.ws + A.wl.counter_off) + b;
        const unsigned long long old = atomic_add_acq_rel(word, inc);  // releases the slot just written
        s_word = old + inc;
        s_last = (old & ((1ull << SPEC_COUNT_BITS) - 1ull)) == (unsigned long long)K ? 1 : 0;  // K + 1 positions
    }
    __syncthreads();
    // Peers only ever push into this CTA's inbox, and the last exchange of the position
    // (the same sequence in every CTA of the cluster) completed on this CTA's own
    // barrier, so nothing is written into its shared memory any more: CTAs may leave now.
    if (g != reporter || s_last == 0) return;
    // thread 0's acquiring add made every position's slot writes visible to it; the
    // barrier above carries that to the rest of the CTA
    spec_finish(A, b, tokens_bad, s_word);
}


size_t spec_workspace_bytes(int B, int K, int V, int G) {
    (void)V;
    (void)G;
    return spec_ws_layout(B, K).total;
}

size_t spec_smem_bytes(int V, int G, int tsz, int dsz, int* t_bytes, int* d_bytes) {
    const size_t nvec = (size_t)(V + VEC - 1) / VEC, cmax = ((nvec + G - 1) / G) * VEC;
    const size_t tb = (cmax * tsz + 15) & ~(size_t)15, db = (cmax * dsz + 15) & ~(size_t)15;
    if (t_bytes) *t_bytes = (int)tb;
    if (d_bytes) *d_bytes = (int)db;
    return STAGE_HEADER + tb + db + draw_smem_bytes(V, G);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_spec_t(const ChainArgs& a, void* ws, int G, cudaStream_t stream) {
    auto kern = chain_spec_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    SpecArgs A;
    A.a = a;
    A.ws = reinterpret_cast<unsigned char*>(ws);
    A.wl = spec_ws_layout(a.B, a.K);
    const size_t smem = spec_smem_bytes(a.V, G, TDT == DT_BF16 ? 2 : 4, DDT == DT_BF16 ? 2 : 4, &A.t_bytes, &A.d_bytes);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int maxc = 0;  // 0 when the shared memory does not fit: the caller takes another kernel
    const cudaError_t e = cache.max_cluster((const void*)kern, cfg, &maxc);
    if (e != cudaSuccess) return e;
    if (maxc < G) return cudaErrorInvalidClusterSize;
    cfg.gridDim = dim3((unsigned)G, (unsigned)(a.K + 1), (unsigned)a.B);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, A);
}

cudaError_t launch_chain_spec(const ChainArgs& a, void* ws, int tdt, int ddt, int dk, int G, cudaStream_t stream) {
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_chain_spec_t<DT_BF16, DT_F32, DK_PROBS>(a, ws, G, stream);
        return launch_chain_spec_t<DT_F32, DT_F32, DK_PROBS>(a, ws, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_chain_spec_t<DT_BF16, DT_BF16, DK_LOGITS>(a, ws, G, stream);
        return launch_chain_spec_t<DT_BF16, DT_F32, DK_LOGITS>(a, ws, G, stream);
    }
    if (ddt == DT_BF16) return launch_chain_spec_t<DT_F32, DT_BF16, DK_LOGITS>(a, ws, G, stream);
    return launch_chain_spec_t<DT_F32, DT_F32, DK_LOGITS>(a, ws, G, stream);
}

}  // namespace sv
