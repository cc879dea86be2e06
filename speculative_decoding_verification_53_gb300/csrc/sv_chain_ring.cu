// sv_chain_ring.cu -- chain verify for large batches: every batch row resident at once,
// each row's vocabulary streamed through a small shared-memory ring.
//
// The rule is the one of sv_chain.cu ("[논문 리뷰] Fast Inference from Transformers
// via Speculative Decoding", section 2, Step 3; "Speculative Decoding and EAGLE",
// section "정확성 규칙"): positions left to right, x_k kept with probability
// min(1, p_k(x_k)/q_k(x_k)), the first rejection drawing from (p_k - q_k)+, the bonus
// token from p_K, greedy rows comparing with the argmax.
//
// Why this layout.  A verify row is a serial chain: position k+1 is read only once
// position k is decided, and a large batch has many such chains.  Staging a whole
// position on chip (sv_chain_staged.cu) takes about 600 KB of shared memory per row at
// V = 152064, so only a few dozen rows fit at once and HBM idles while each of them
// computes and exchanges.  Here a row's chunk is streamed instead: a cluster of G
// small CTAs per row (128 threads, a ring of three 2048-element stages of target and
// draft each, about 28 KB of shared memory) keeps every row of a batch of a few
// hundred resident, so while some rows exchange statistics, draw or wait for a
// decision, the others keep their bulk copies in flight.
//
// Measured, this loses to the staged walk (B = 256, K = 8, V = 152064: 212 against
// 146 us at T = 0.7): a CTA of four warps alone on its SM streams and reduces only
// about 10 GB/s, so once most rows have finished, the long chains that remain crawl.
// It runs only when requested (SPEC_VERIFY_PATH=ring) and is kept, tested, as the
// record of that design.
//
// Per position k, every CTA streams its chunk [lo, hi) of the target row (and of the
// draft-logit row) through the ring, reducing online to (max, sum of exp2) per row
// (greedy rows: the argmax); the cluster combines the partials through distributed
// shared memory; every CTA loads l_k(x_k) (and the draft value at x_k) itself and
// takes the same decision.  At the first rejection (or the bonus position) the chunk
// of that position is streamed once more, now from L2, to sum the residual weights per
// 256-element tile; the inverse-CDF search over the tile sums is the one of
// sv_common.cuh (cluster_draw_from_tiles).  Rows are 16-byte aligned (bulk copies).
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int RING_NT = 128;            // threads per CTA
constexpr int RING_NW = RING_NT / 32;   // warps per CTA
constexpr int RING_PE = 2048;           // elements per ring stage (8 tiles of 256)
constexpr int RING_TILES = RING_PE / TILE;
constexpr int RING_TPW = RING_TILES / RING_NW;  // tiles per warp per stage
constexpr int RING_MAX_G = 8;
constexpr int RING_HEADER = 128;        // the stages' mbarriers
static_assert(RING_TILES % RING_NW == 0, "whole tiles per warp");

// Exchange state of a ring CTA (the fields the draw's exchange in sv_common.cuh uses,
// sized for four warps).
struct RingScratch {
    uint64_t xbar[2];
    struct {
        float4 part[2][RING_MAX_G][RING_NW];
        float2 zf[2][MAX_CLUSTER];
    } inbox;
    float bf[8];
    int bi[8];
};

// Weights of the draw read from global memory, with the arithmetic of the ring's tile
// pass (so the owner's search sees the values the tile sums were made of).  RES: the
// residual max(0, p - q); otherwise p.
template <int TDT, int DDT, int DK, bool RES>
struct RingWeights {
    static constexpr int kTilesInFlight = 4;
    const void* trow;
    const void* drow;
    float c, mtc, inv_st, mdc, inv_sd;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC], d[VEC];
        load8<TDT>(trow, e0, hi, true, neg_inf(), l);
        if (RES) load8<DDT>(drow, e0, hi, true, DK == DK_LOGITS ? neg_inf() : 0.f, d);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float p = __fmul_rn(ex2(fmaf(l[j], c, -mtc)), inv_st);
            if (RES) {
                const float q = (DK == DK_LOGITS) ? __fmul_rn(ex2(fmaf(d[j], c, -mdc)), inv_sd) : d[j];
                w[j] = fmaxf(__fsub_rn(p, q), 0.f);
            } else {
                w[j] = p;
            }
        }
    }
};

// Online (max, sum 2^((x - max) c)) over 16 values held by a thread; vm is their maximum
// (NaN when one is NaN).
__device__ __forceinline__ void lse_add16(LSE& acc, float& mc, const float x[2][VEC], float vm, float c) {
    if (vm != vm) acc.bad = 1;
    if (vm > acc.m) {
        acc.s *= ex2((acc.m - vm) * c);
        acc.m = vm;
        mc = vm * c;
    }
    if (acc.m > neg_inf()) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            s0 += ex2(fmaf(x[i][0], c, -mc)) + ex2(fmaf(x[i][4], c, -mc));
            s1 += ex2(fmaf(x[i][1], c, -mc)) + ex2(fmaf(x[i][5], c, -mc));
            s2 += ex2(fmaf(x[i][2], c, -mc)) + ex2(fmaf(x[i][6], c, -mc));
            s3 += ex2(fmaf(x[i][3], c, -mc)) + ex2(fmaf(x[i][7], c, -mc));
        }
        acc.s += (s0 + s1) + (s2 + s3);
    }
}

// Eight staged values at element e of a stage buffer (padded beyond n) and their maximum.
template <int DT>
__device__ __forceinline__ float ring_load8(const unsigned char* buf, int e, int n, float pad, float x[VEC]) {
    if (DT == DT_BF16 && e + VEC <= n) {
        const uint4 v = *reinterpret_cast<const uint4*>(buf + (size_t)e * 2);
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
        const uint32_t m = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    }
    smem_load8<DT>(buf, e, n, pad, x);
    return vmax8(x);
}

// Cluster combine of the position's statistics: (max, sum) of the target row and, when
// TWO, of the draft row.  Lanes 0..G-1 of every warp push the warp's partials into CTA
// `lane`'s inbox; warp 0 waits for its own inbox (bounded) and combines the G * 4
// partials, one per lane.  Flags travel as NaN sums (flagged_sum); a wait that gives up
// flags both rows BAD_TIMEOUT.
template <bool TWO>
__device__ __forceinline__ void ring_stats(LSE& t, LSE& d, float c, RingScratch& sc, int& phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = (int)cluster_size(), me = (int)cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, (uint32_t)(G * RING_NW) * 16u);
    if (TWO) {
        lse2_warp_reduce(t, d, c);
    } else {
        lse_warp_reduce(t, c);
    }
    if (lane < G) {
        const float4 v = make_float4(t.m, flagged_sum(t), TWO ? d.m : neg_inf(), TWO ? flagged_sum(d) : 0.f);
        st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][warp], (uint32_t)lane), v, xchg_bar(sc, phase, (uint32_t)lane));
    }
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        const int E = G * RING_NW;  // at most 32 partials: one per lane
        const float4 v = lane < E ? sc.inbox.part[buf][lane / RING_NW][lane % RING_NW]
                                  : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
        float Mt = v.x, Md = v.z;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
            if (TWO) Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, o));
        }
        float St = (v.x > neg_inf() && v.y == v.y) ? v.y * ex2((v.x - Mt) * c) : 0.f;
        float Sd = (TWO && v.z > neg_inf() && v.w == v.w) ? v.w * ex2((v.z - Md) * c) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            St += __shfl_xor_sync(0xffffffffu, St, o);
            if (TWO) Sd += __shfl_xor_sync(0xffffffffu, Sd, o);
        }
        const int bt = (int)__reduce_or_sync(0xffffffffu, (unsigned)sum_flags(v.y)) | (ok ? 0 : BAD_TIMEOUT);
        const int bd = (int)__reduce_or_sync(0xffffffffu, (unsigned)sum_flags(v.w)) | (ok ? 0 : BAD_TIMEOUT);
        if (lane == 0) {
            sc.bf[0] = Mt; sc.bf[1] = St; sc.bf[2] = Md; sc.bf[3] = Sd;
            sc.bi[0] = bt; sc.bi[1] = bd;
        }
    }
    __syncthreads();
    t = LSE{sc.bf[0], sc.bf[1], sc.bi[0]};
    d = LSE{sc.bf[2], sc.bf[3], TWO ? sc.bi[1] : 0};
    __syncthreads();
    ++phase;
}

__device__ __forceinline__ ArgMax ring_argmax(ArgMax a, RingScratch& sc, int& phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = (int)cluster_size(), me = (int)cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, (uint32_t)(G * RING_NW) * 16u);
    argmax_warp_reduce(a);
    if (lane < G)
        st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][warp], (uint32_t)lane),
                    make_float4(a.v, __int_as_float(a.i), __int_as_float(a.bad), 0.f), xchg_bar(sc, phase, (uint32_t)lane));
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        ArgMax x{neg_inf(), 0x7fffffff, ok ? 0 : BAD_TIMEOUT};
        if (lane < G * RING_NW) {
            const float4 v = sc.inbox.part[buf][lane / RING_NW][lane % RING_NW];
            argmax_merge(x, ArgMax{v.x, __float_as_int(v.y), __float_as_int(v.z)});
        }
        argmax_warp_reduce(x);
        if (lane == 0) {
            sc.bf[0] = x.v;
            sc.bi[0] = x.i;
            sc.bi[1] = x.bad;
        }
    }
    __syncthreads();
    ArgMax r{sc.bf[0], sc.bi[0], sc.bi[1]};
    __syncthreads();
    ++phase;
    return r;
}

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(RING_NT, 8) chain_ring_kernel(const ChainArgs a, const RingLayout L) {
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(dsm);  // one mbarrier per stage
    unsigned char* stages = dsm + RING_HEADER;
    float* tile_sum = reinterpret_cast<float*>(stages + (size_t)L.nstage * L.stage_bytes);
    __shared__ RingScratch sc;
    __shared__ int s_tok[MAX_K];
    __shared__ float s_r[MAX_K + 1], s_u[MAX_K + 1], s_ap[MAX_K];
    __shared__ float s_g[2];  // l_k(x_k) and the draft's value at x_k
    const int G = (int)cluster_size(), g = (int)cluster_rank();
    const int b = blockIdx.y;
    const int K = a.K, V = a.V;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int lo, hi;
    chunk_range(V, g, G, lo, hi);
    const int n = hi - lo;
    const int npieces = (n + RING_PE - 1) / RING_PE;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const unsigned char* tbase = reinterpret_cast<const unsigned char*>(a.target) + (size_t)b * (K + 1) * V * tsz;
    const unsigned char* dbase = reinterpret_cast<const unsigned char*>(a.draft) + (size_t)b * K * V * dsz;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L.nstage; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // the Philox blocks (kernel parameters only) on warps 1.., before the dependency wait
    for (int k = (int)threadIdx.x - 32; k >= 0 && k <= K; k += RING_NT - 32)
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, s_r[k], s_u[k]);
    xchg_init_arrive(sc);
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    const float T = a.temperature ? a.temperature[b] : 0.f;
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool draft_rows = !greedy && DK == DK_LOGITS;  // draft-logit rows are streamed with the target rows

    // Ring bookkeeping: stage number gs (counted over the whole kernel) lives in slot
    // gs % nstage and completes phase (gs / nstage) of that slot's barrier.  A pass over
    // position k streams pieces 0..npieces-1 of the chunk (target, plus the draft row
    // when `with_d`); thread 0 issues a piece once its slot has been read.
    uint32_t gs = 0;
    auto issue = [&](int k, bool with_d, int j, uint32_t gsj) {
        const int s = (int)(gsj % (uint32_t)L.nstage);
        const int e0 = lo + j * RING_PE;
        const int cnt = min(RING_PE, hi - e0);
        unsigned char* st = stages + (size_t)s * L.stage_bytes;
        fence_proxy_async();
        mbar_arrive_expect_tx(&full[s], (uint32_t)cnt * (tsz + (with_d ? dsz : 0)));
        bulk_g2s(st, tbase + ((size_t)k * V + e0) * tsz, (uint32_t)cnt * tsz, &full[s]);
        if (with_d) bulk_g2s(st + L.t_bytes, dbase + ((size_t)k * V + e0) * dsz, (uint32_t)cnt * dsz, &full[s]);
    };
    auto issue_first = [&](int k, bool with_d) {
        if (threadIdx.x == 0)
            for (int j = 0; j < L.nstage && j < npieces; ++j) issue(k, with_d, j, gs + (uint32_t)j);
    };
    // Waits for piece j of the current pass and returns its stage; `fail` collects waits
    // that gave up.
    auto wait_piece = [&](int j, int& fail) -> const unsigned char* {
        const uint32_t gsj = gs + (uint32_t)j;
        const int s = (int)(gsj % (uint32_t)L.nstage);
        if (!mbar_wait_bounded(&full[s], (gsj / (uint32_t)L.nstage) & 1u)) fail = 1;
        return stages + (size_t)s * L.stage_bytes;
    };
    // After piece j has been read by every thread: refill its slot with piece j + nstage.
    auto release_piece = [&](int k, bool with_d, int j) {
        __syncthreads();
        if (threadIdx.x == 0 && j + L.nstage < npieces) issue(k, with_d, j + L.nstage, gs + (uint32_t)(j + L.nstage));
    };

    issue_first(0, draft_rows && K > 0);  // position 0 goes out before the token checks
    int tok_bad = 0;
    if ((int)threadIdx.x < K) {
        const int x = a.tokens[(size_t)b * K + threadIdx.x];
        s_tok[threadIdx.x] = x;
        s_ap[threadIdx.x] = -1.f;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    for (int k = (int)threadIdx.x + RING_NT; k < K; k += RING_NT) {
        const int x = a.tokens[(size_t)b * K + k];
        s_tok[k] = x;
        s_ap[k] = -1.f;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    bool invalid = __syncthreads_or(tok_bad) != 0;
    xchg_ready();

    // tmo: some wait of the row gave up (this CTA's, or a peer's flag seen in an exchange)
    int phase = 0, j = -1, final_tok = -1, writer = 0, tmo = 0;
    if (invalid) {  // the copies of position 0 are in flight: let them land before leaving
        int f = 0;
        for (int p = 0; p < L.nstage && p < npieces; ++p) (void)wait_piece(p, f);
        gs += (uint32_t)npieces;
    }
    for (int k = 0; k <= K && !invalid; ++k) {
        const bool with_d = draft_rows && k < K;
        if (k > 0) issue_first(k, with_d);
        const int x = k < K ? s_tok[k] : -1;
        // the values at x_k: one direct load each, in flight during the pass
        float gx_t = 0.f, gx_d = 0.f;
        if (!greedy && k < K && threadIdx.x == 0) {
            gx_t = load_one<TDT>(tbase + (size_t)k * V * tsz, x);
            gx_d = DK == DK_LOGITS ? load_one<DDT>(dbase + (size_t)k * V * dsz, x)
                                   : load_one<DT_F32>(dbase + (size_t)k * V * dsz, x);
        }
        int fail = 0;
        if (greedy) {
            ArgMax am{neg_inf(), 0x7fffffff, 0};
            for (int p = 0; p < npieces; ++p) {
                const unsigned char* st = wait_piece(p, fail);
                const int cnt = min(RING_PE, n - p * RING_PE);
#pragma unroll
                for (int i = 0; i < RING_TPW; ++i) {
                    const int e = (warp + i * RING_NW) * TILE + lane * VEC;
                    if (e < cnt) {
                        float xv[VEC];
                        const float vm = ring_load8<TDT>(st, e, cnt, neg_inf(), xv);
                        if (vm != vm) am.bad = 1;
                        if (vm > am.v) {  // strictly greater: the lower index keeps ties
                            int jj = 0;
#pragma unroll
                            for (int t = VEC - 1; t >= 0; --t)
                                if (xv[t] == vm) jj = t;
                            am.v = vm;
                            am.i = lo + p * RING_PE + e + jj;
                        }
                    }
                }
                release_piece(k, false, p);
            }
            gs += (uint32_t)npieces;
            if (__syncthreads_or(fail)) am.bad |= BAD_TIMEOUT;
            am = ring_argmax(am, sc, phase);
            if (am.bad & BAD_TIMEOUT) tmo = 1;
            if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) { invalid = true; break; }
            if (k < K && x == am.i) {
                if (threadIdx.x == 0) s_ap[k] = 1.f;
                continue;
            }
            if (k < K && threadIdx.x == 0) s_ap[k] = 0.f;
            j = k;
            final_tok = am.i;
            writer = 0;
            break;
        }
        // ---- sampling row: streaming statistics of the target (and draft-logit) row
        LSE ts{neg_inf(), 0.f, 0}, ds{neg_inf(), 0.f, 0};
        float tmc = 0.f, dmc = 0.f;
        for (int p = 0; p < npieces; ++p) {
            const unsigned char* st = wait_piece(p, fail);
            const int cnt = min(RING_PE, n - p * RING_PE);
            float xt[RING_TPW][VEC];
            float vt = neg_inf();
#pragma unroll
            for (int i = 0; i < RING_TPW; ++i) {
                const int e = (warp + i * RING_NW) * TILE + lane * VEC;
                if (e < cnt) {
                    vt = fmax_nan(vt, ring_load8<TDT>(st, e, cnt, neg_inf(), xt[i]));
                } else {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) xt[i][q] = neg_inf();
                }
            }
            lse_add16(ts, tmc, xt, vt, c);
            if (with_d) {
                float xd[RING_TPW][VEC];
                float vd = neg_inf();
#pragma unroll
                for (int i = 0; i < RING_TPW; ++i) {
                    const int e = (warp + i * RING_NW) * TILE + lane * VEC;
                    if (e < cnt) {
                        vd = fmax_nan(vd, ring_load8<DDT>(st + L.t_bytes, e, cnt, neg_inf(), xd[i]));
                    } else {
#pragma unroll
                        for (int q = 0; q < VEC; ++q) xd[i][q] = neg_inf();
                    }
                }
                lse_add16(ds, dmc, xd, vd, c);
            }
            release_piece(k, with_d, p);
        }
        gs += (uint32_t)npieces;
        if (__syncthreads_or(fail)) ts.bad |= BAD_TIMEOUT;
        if (threadIdx.x == 0) {
            s_g[0] = gx_t;
            s_g[1] = gx_d;
        }
        ring_stats<DK == DK_LOGITS>(ts, ds, c, sc, phase);
        if ((ts.bad | ds.bad) & BAD_TIMEOUT) tmo = 1;
        if (row_bad_s(ts) || (with_d && row_bad_s(ds))) { invalid = true; break; }
        const float inv_st = 1.f / ts.s;
        const float inv_sd = with_d ? 1.f / ds.s : 0.f;
        bool draw = true;
        if (k < K) {
            const float px = ex2((s_g[0] - ts.m) * c) * inv_st;
            float qx;
            if (DK == DK_LOGITS) {
                qx = ex2((s_g[1] - ds.m) * c) * inv_sd;
            } else {
                qx = s_g[1];
                if (!(qx >= 0.f) || qx == pos_inf()) { invalid = true; break; }
            }
            const float ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
            if (threadIdx.x == 0) s_ap[k] = fminf(ratio, 1.f);
            draw = !(s_r[k] < ratio);
        }
        if (!draw) continue;
        // ---- the draw at k: the residual (p_k - q_k)+, or p_K for the bonus token.  The
        // chunk is streamed once more (from L2: it was read just before) and each warp
        // sums the weights of its 256-element tiles.
        const bool res = k < K;  // draft row needed (logits or probabilities)
        issue_first(k, res);
        const float mtc = ts.m * c, mdc = ds.m * c;
        int dfail = 0;
        for (int p = 0; p < npieces; ++p) {
            const unsigned char* st = wait_piece(p, dfail);
            const int cnt = min(RING_PE, n - p * RING_PE);
#pragma unroll
            for (int i = 0; i < RING_TPW; ++i) {
                const int tile = warp + i * RING_NW;
                const int e = tile * TILE + lane * VEC;
                float s = 0.f;
                if (e < cnt) {
                    float l[VEC];
                    smem_load8<TDT>(st, e, cnt, neg_inf(), l);
                    if (res) {
                        float d[VEC];
                        if (DK == DK_LOGITS) {
                            smem_load8<DDT>(st + L.t_bytes, e, cnt, neg_inf(), d);
                        } else {
                            smem_load8<DT_F32>(st + L.t_bytes, e, cnt, 0.f, d);
                        }
#pragma unroll
                        for (int q = 0; q < VEC; ++q) {
                            const float pp = __fmul_rn(ex2(fmaf(l[q], c, -mtc)), inv_st);
                            const float qq =
                                (DK == DK_LOGITS) ? __fmul_rn(ex2(fmaf(d[q], c, -mdc)), inv_sd) : d[q];
                            s += fmaxf(__fsub_rn(pp, qq), 0.f);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < VEC; ++q) s += __fmul_rn(ex2(fmaf(l[q], c, -mtc)), inv_st);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) tile_sum[p * RING_TILES + tile] = s;
            }
            release_piece(k, res, p);
        }
        gs += (uint32_t)npieces;
        dfail = __syncthreads_or(dfail);
        const void* trow = tbase + (size_t)k * V * tsz;
        const void* drow = res ? (const void*)(dbase + (size_t)k * V * dsz) : nullptr;
        DrawResult d;
        if (res) {
            const RingWeights<TDT, DDT, DK, true> rw{trow, drow, c, mtc, inv_st, mdc, inv_sd};
            d = cluster_draw_from_tiles(rw, lo, hi, s_u[k], tile_sum, sc, phase, dfail);
            if (!d.failed && d.owner < 0) {  // the residual has no mass: draw from p_k
                const RingWeights<TDT, DDT, DK, false> pw{trow, nullptr, c, mtc, inv_st, 0.f, 0.f};
                d = cluster_draw(pw, lo, hi, s_u[k], tile_sum, sc, phase);
            }
        } else {
            const RingWeights<TDT, DDT, DK, false> pw{trow, nullptr, c, mtc, inv_st, 0.f, 0.f};
            d = cluster_draw_from_tiles(pw, lo, hi, s_u[k], tile_sum, sc, phase, dfail);
        }
        if (d.failed) tmo = 1;
        if (d.failed || d.owner < 0) { invalid = true; break; }
        j = k;
        final_tok = d.token;
        writer = d.owner;
        break;
    }
    __syncthreads();
    if (invalid) writer = 0;
    if (g == writer) {
        int32_t* ot = a.out_tokens + (size_t)b * (K + 1);
        for (int i = threadIdx.x; i <= K; i += RING_NT)
            ot[i] = invalid ? -1 : (i < j ? s_tok[i] : (i == j ? final_tok : -1));
        if (a.out_accept_prob)
            for (int i = threadIdx.x; i < K; i += RING_NT)
                a.out_accept_prob[(size_t)b * K + i] = invalid ? -1.f : s_ap[i];
        if (threadIdx.x == 0) a.out_count[b] = invalid ? (tmo ? SV_COUNT_TIMEOUT : 0) : j + 1;
    }
    // Leave together: a CTA whose bounded wait gave up may have taken another branch than
    // its peers, which could still push an exchange into its shared memory.  Every wait
    // before this barrier is bounded, so every CTA of the cluster reaches it.  A CTA that
    // saw a timeout then marks the row (after the barrier, so after any other writer).
    cluster_sync_all();
    if (tmo && threadIdx.x == 0) a.out_count[b] = SV_COUNT_TIMEOUT;
}

size_t ring_smem_bytes(const RingLayout& L, int V, int G) {
    const int nvec = (V + VEC - 1) / VEC, cap = ((nvec + G - 1) / G) * VEC;
    const int npieces = (cap + RING_PE - 1) / RING_PE;
    return RING_HEADER + (size_t)L.nstage * L.stage_bytes + (size_t)npieces * RING_TILES * sizeof(float);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_ring_t(const ChainArgs& a, const RingLayout& L, int G, cudaStream_t stream) {
    auto kern = chain_ring_kernel<TDT, DDT, DK>;
    static KernelLaunchCache cache;
    const size_t smem = ring_smem_bytes(L, a.V, G);
    int max_cluster = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(RING_NT, 1, 1);
    cfg.stream = stream;
    cfg.dynamicSmemBytes = smem;
    const cudaError_t e = cache.max_cluster((const void*)kern, cfg, &max_cluster);
    if (e != cudaSuccess) return e;
    if (max_cluster < G) return cudaErrorInvalidClusterSize;  // caller takes another kernel
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

cudaError_t launch_chain_ring(const ChainArgs& a, const RingLayout& L, int tdt, int ddt, int dk, int G,
                              cudaStream_t stream) {
    if (G < 1 || G > RING_MAX_G) return cudaErrorInvalidClusterSize;
    if (dk == DK_PROBS) {
        if (tdt == DT_BF16) return launch_chain_ring_t<DT_BF16, DT_F32, DK_PROBS>(a, L, G, stream);
        return launch_chain_ring_t<DT_F32, DT_F32, DK_PROBS>(a, L, G, stream);
    }
    if (tdt == DT_BF16) {
        if (ddt == DT_BF16) return launch_chain_ring_t<DT_BF16, DT_BF16, DK_LOGITS>(a, L, G, stream);
        return launch_chain_ring_t<DT_BF16, DT_F32, DK_LOGITS>(a, L, G, stream);
    }
    if (ddt == DT_BF16) return launch_chain_ring_t<DT_F32, DT_BF16, DK_LOGITS>(a, L, G, stream);
    return launch_chain_ring_t<DT_F32, DT_F32, DK_LOGITS>(a, L, G, stream);
}

}  // namespace sv
