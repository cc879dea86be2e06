// sv_chain_spec.cu -- position-parallel chain verify for small batches.
//
// The rule is the one of sv_chain.cu ("[논문 리뷰] Fast Inference from
// Transformers via Speculative Decoding", section 2, Step 3; "Speculative
// Decoding and EAGLE", section "정확성 규칙"), evaluated in another order.  For a
// small batch the left-to-right walk over positions is latency-bound (one
// cluster exchange per position), so here every position k of every batch row b
// gets its own cluster of G CTAs at once:
//   1. the cluster stages its chunk of target row k (and draft row k), computes
//      the softmax statistics and the acceptance test of x_k (greedy: the argmax),
//   2. speculatively prepares the draw at k as if k were the first rejection:
//      per-tile sums of the residual (p_k - q_k)+ (and of p_k, the zero-mass
//      fallback; p_K for the bonus position), written to the workspace,
//   3. publishes a per-position record and counts itself in with one atomic;
// the last CTA to arrive for batch row b (no CTA ever waits for another) finds
// the first rejection j from the records, picks the CTA chunk and the 256-entry
// tile that hold u_j * Z from the published sums, recomputes that tile's weights
// from global memory and writes the outputs.  The results are those of the
// left-to-right rule; only work is done speculatively, and reads of positions
// past the first rejection are the price of the shorter critical path.
#include "sv_stage.cuh"
#include "sv_internal.h"

namespace sv {

// Per (row, position) record published by the cluster's rank-0 CTA.
struct SpecRec {
    float tm, ts, dm, ds;  // target / draft statistics (max, sum of exp2)
    float ratio;           // p_k(x_k) / q_k(x_k) (sampling rows)
    float u;               // draw uniform of slot k
    int flags;             // SPEC_* bits
    int argmax;            // greedy rows: argmax of target row k
};

constexpr int SPEC_BAD = 1;     // the position's rows (or q(x_k)) are invalid
constexpr int SPEC_ACCEPT = 2;  // sampling: r_k < ratio; greedy: x_k == argmax

// Workspace carve-up (all offsets 256-byte aligned), identical on host and device.
struct SpecWsLayout {
    size_t counter_off, rec_off, z_off, tile_off, total;
    int ntiles;  // tile-sum slots per CTA chunk
};

__host__ __device__ inline size_t spec_align(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline SpecWsLayout spec_ws_layout(int B, int K, int V, int G) {
    SpecWsLayout L;
    const size_t nvec = (size_t)(V + VEC - 1) / VEC, cmax = ((nvec + G - 1) / G) * VEC;
    L.ntiles = (int)((cmax + TILE - 1) / TILE);
    const size_t P = (size_t)B * (K + 1);
    L.counter_off = 0;
    L.rec_off = spec_align(L.counter_off + (size_t)B * sizeof(unsigned));
    L.z_off = spec_align(L.rec_off + P * sizeof(SpecRec));
    L.tile_off = spec_align(L.z_off + P * G * 2 * sizeof(float));
    L.total = spec_align(L.tile_off + P * G * 2 * (size_t)L.ntiles * sizeof(float));
    return L;
}

struct SpecArgs {
    ChainArgs a;
    unsigned char* ws;
    SpecWsLayout wl;
    int t_bytes;  // shared-memory offset of the draft chunk
    int d_bytes;  // bytes reserved for the draft chunk (tile sums follow)
    int fin_off;  // shared-memory offset of the finishing step's chunk totals
};

// Residual and plain-p weights of 8 staged elements, with rounding pinned by _rn
// intrinsics so that the finishing CTA, recomputing one tile from global memory,
// reproduces the sums the position's cluster published.
template <int DK>
__device__ __forceinline__ void spec_weights8(const float l[VEC], const float d[VEC], float c, float mt, float inv_st,
                                              float md, float inv_sd, float w_res[VEC], float w_p[VEC]) {
    const float mtc = __fmul_rn(mt, c), mdc = __fmul_rn(md, c);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const float p = __fmul_rn(ex2(__fmaf_rn(l[j], c, -mtc)), inv_st);
        const float q = (DK == DK_LOGITS) ? __fmul_rn(ex2(__fmaf_rn(d[j], c, -mdc)), inv_sd) : d[j];
        w_p[j] = p;
        w_res[j] = fmaxf(__fsub_rn(p, q), 0.f);
    }
}


// Finishing step for batch row b, run by the last CTA to arrive (global memory only).
template <int TDT, int DDT, int DK>
__device__ void spec_finish(const SpecArgs& A, int b, bool greedy, bool tok_bad, const int* s_tok, SpecRec* s_rec,
                            int* s_int, float* s_z);

template <int TDT, int DDT, int DK>
__global__ void __launch_bounds__(NT) chain_spec_kernel(const SpecArgs A) {
    const ChainArgs& a = A.a;
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t* tbar = reinterpret_cast<uint64_t*>(dsm);
    uint64_t* dbar = tbar + 1;
    unsigned char* tb = dsm + STAGE_HEADER;  // target chunk of row (b, k)
    unsigned char* db = tb + A.t_bytes;      // draft chunk (logits or probabilities)
    float* s_tile = reinterpret_cast<float*>(db + A.d_bytes);  // [2][ntiles] tile sums of this chunk
    __shared__ BlockScratch sc;
    __shared__ int s_tok[MAX_K];
    __shared__ SpecRec s_rec[MAX_K + 1];
    __shared__ float s_flt[4];
    __shared__ int s_int[4];

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
    if (threadIdx.x == 0) {
        mbar_init(tbar, 1);
        mbar_init(dbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(tbar, (uint32_t)n * tsz);
        if (n) bulk_g2s(tb, trow + (size_t)lo * tsz, (uint32_t)n * tsz, tbar);
        if (has_draft_row) {
            mbar_arrive_expect_tx(dbar, (uint32_t)n * dsz);
            if (n) bulk_g2s(db, drow + (size_t)lo * dsz, (uint32_t)n * dsz, dbar);
        }
    }
    int tok_bad = 0;
    for (int i = threadIdx.x; i < K; i += NT) {
        const int x = a.tokens[(size_t)b * K + i];
        s_tok[i] = x;
        if (x < 0 || x >= V) tok_bad = 1;
    }
    if (threadIdx.x == 32) {  // warp 1: the Philox block of slot k (unused on greedy rows)
        float r, u;
        slot_uniforms(a.seed, a.offset, (uint64_t)b, (uint64_t)k, r, u);
        s_flt[0] = r;
        s_flt[1] = u;
    }
    const float T = a.temperature ? a.temperature[b] : 0.f;
    const bool greedy = !(T > 0.f);
    const float c = greedy ? 0.f : LOG2E / T;
    const bool tokens_bad = __syncthreads_or(tok_bad) != 0;

    // 2. statistics of row k, the acceptance test of x_k
    bool ok = mbar_wait_bounded(tbar, 0);
    if (has_draft_row) ok = mbar_wait_bounded(dbar, 0) && ok;
    const int fail = __syncthreads_or(!ok);
    const int x = (k < K && !tokens_bad) ? s_tok[k] : -1;
    int phase = 0, flags = 0, amax = -1;
    float ratio = 0.f;
    PosStats ps{};
    if (greedy) {
        ArgMax am = smem_thread_argmax<TDT>(tb, n, lo);
        if (fail) am.bad = 1;
        am = cluster_argmax(am, sc, phase);
        if (am.bad || !(am.v > neg_inf()) || am.v == pos_inf()) flags |= SPEC_BAD;
        if (k < K && x == am.i) flags |= SPEC_ACCEPT;
        amax = am.i;
    } else {
        LSE ts = smem_thread_lse<TDT>(tb, n, c);
        LSE ds{neg_inf(), 0.f, 0};
        if (DK == DK_LOGITS && k < K) ds = smem_thread_lse<DDT>(db, n, c);
        if (fail) ts.bad = 1;
        float tx = 0.f, dx = 0.f;
        int has = 0;
        if (threadIdx.x == 0 && x >= lo && x < hi) {
            tx = smem_elem<TDT>(tb, x - lo);
            dx = (DK == DK_LOGITS) ? smem_elem<DDT>(db, x - lo) : smem_elem<DT_F32>(db, x - lo);
            has = 1;
        }
        ps = cluster_pos_stats(ts, ds, c, tx, dx, has, sc, phase);
        bool bad = row_bad_s(ps.t) || (DK == DK_LOGITS && k < K && row_bad_s(ps.d));
        const float inv_st = 1.f / ps.t.s;
        const float inv_sd = (DK == DK_LOGITS && k < K) ? 1.f / ps.d.s : 0.f;
        if (k < K && !bad) {
            const float px = ex2((ps.tx - ps.t.m) * c) * inv_st;
            const float qx = (DK == DK_LOGITS) ? ex2((ps.dx - ps.d.m) * c) * inv_sd : ps.dx;
            if (DK == DK_PROBS && (!(qx >= 0.f) || qx == pos_inf())) bad = true;
            ratio = qx > 0.f ? px / qx : (px > 0.f ? pos_inf() : 0.f);
            if (s_flt[0] < ratio) flags |= SPEC_ACCEPT;
        }
        if (bad) flags |= SPEC_BAD;
        // 3. the draw at k, prepared as if k were the first rejection: per-tile sums of the
        // residual (set 0) and of p (set 1; at the bonus position set 0 is p itself)
        if (!bad && !tokens_bad) {
            const int ntiles = (n + TILE - 1) / TILE;
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            float* gt = reinterpret_cast<float*>(A.ws + A.wl.tile_off) +
                        ((((size_t)b * (K + 1) + k) * G + g) * 2) * A.wl.ntiles;
            for (int t0 = warp; t0 < ntiles; t0 += 2 * NW) {  // two tiles per warp step, for overlap
                float sr[2] = {0.f, 0.f}, sp[2] = {0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = (t0 + h * NW) * TILE + lane * VEC;  // chunk-local
                    float l[VEC], d[VEC], wr[VEC], wp[VEC];
                    smem_load8<TDT>(tb, e, n, neg_inf(), l);
                    if (k < K) {
                        smem_load8<DDT>(db, e, n, DK == DK_LOGITS ? neg_inf() : 0.f, d);
                    } else {
#pragma unroll
                        for (int q = 0; q < VEC; ++q) d[q] = DK == DK_LOGITS ? neg_inf() : 0.f;
                    }
                    spec_weights8<DK>(l, d, c, ps.t.m, inv_st, ps.d.m, inv_sd, wr, wp);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) {
                        sr[h] += wr[q];
                        sp[h] += wp[q];
                    }
                    if (k == K) sr[h] = sp[h];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sr[0] += __shfl_xor_sync(0xffffffffu, sr[0], o);
                    sp[0] += __shfl_xor_sync(0xffffffffu, sp[0], o);
                    sr[1] += __shfl_xor_sync(0xffffffffu, sr[1], o);
                    sp[1] += __shfl_xor_sync(0xffffffffu, sp[1], o);
                }
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = t0 + h * NW;
                        if (t < ntiles) {
                            gt[t] = sr[h];
                            gt[A.wl.ntiles + t] = sp[h];
                            s_tile[t] = sr[h];
                            s_tile[ntiles + t] = sp[h];
                        }
                    }
                }
            }
            __syncthreads();
            if (warp == 0) {  // chunk totals in tile order, as the finishing CTA will add them
                float zr = 0.f, zp = 0.f;
                for (int t = lane; t < ntiles; t += 32) {
                    zr += s_tile[t];
                    zp += s_tile[ntiles + t];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    zr += __shfl_xor_sync(0xffffffffu, zr, o);
                    zp += __shfl_xor_sync(0xffffffffu, zp, o);
                }
                if (lane == 0) {
                    float* z = reinterpret_cast<float*>(A.ws + A.wl.z_off) + (((size_t)b * (K + 1) + k) * G + g) * 2;
                    z[0] = zr;
                    z[1] = zp;
                }
            }
        }
    }
    // 4. publish the position record and count this CTA in
    if (g == 0 && threadIdx.x == 0) {
        SpecRec* rec = reinterpret_cast<SpecRec*>(A.ws + A.wl.rec_off) + (size_t)b * (K + 1) + k;
        rec->tm = ps.t.m;
        rec->ts = ps.t.s;
        rec->dm = ps.d.m;
        rec->ds = ps.d.s;
        rec->ratio = ratio;
        rec->u = greedy ? 0.f : s_flt[1];
        rec->flags = flags;
        rec->argmax = amax;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned* counter = reinterpret_cast<unsigned*>(A.ws + A.wl.counter_off) + b;
        const unsigned old = atomicAdd(counter, 1u);
        s_int[0] = (old == (unsigned)((K + 1) * G - 1)) ? 1 : 0;
    }
    __syncthreads();
    const bool last = s_int[0] != 0;
    cluster_sync_all();  // every remote shared-memory read of this cluster is done
    if (!last) return;
    __threadfence();
    spec_finish<TDT, DDT, DK>(A, b, greedy, tokens_bad, s_tok, s_rec, s_int,
                              reinterpret_cast<float*>(dsm + A.fin_off));
}


template <int TDT, int DDT, int DK>
__device__ void spec_finish(const SpecArgs& A, int b, bool greedy, bool tok_bad, const int* s_tok, SpecRec* s_rec,
                            int* s_int, float* s_z) {
    const ChainArgs& a = A.a;
    const int K = a.K, V = a.V, G = (int)cluster_size();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int tsz = TDT == DT_BF16 ? 2 : 4, dsz = DDT == DT_BF16 ? 2 : 4;
    const SpecRec* grec = reinterpret_cast<const SpecRec*>(A.ws + A.wl.rec_off) + (size_t)b * (K + 1);
    for (int i = threadIdx.x; i <= K; i += NT) {  // records written by other SMs: read through L2
        SpecRec r;
        r.tm = __ldcg(&grec[i].tm);
        r.ts = __ldcg(&grec[i].ts);
        r.dm = __ldcg(&grec[i].dm);
        r.ds = __ldcg(&grec[i].ds);
        r.ratio = __ldcg(&grec[i].ratio);
        r.u = __ldcg(&grec[i].u);
        r.flags = __ldcg(&grec[i].flags);
        r.argmax = __ldcg(&grec[i].argmax);
        s_rec[i] = r;
    }
    if (!greedy) {  // every position's chunk totals, in the same round trip as the records
        const float* zall = reinterpret_cast<const float*>(A.ws + A.wl.z_off) + (size_t)b * (K + 1) * G * 2;
        for (int i = threadIdx.x; i < (K + 1) * G * 2; i += NT) s_z[i] = __ldcg(&zall[i]);
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // first rejection (or mismatch); rows read up to it must be valid
        int j = K;
        for (int i = 0; i < K; ++i)
            if (!(s_rec[i].flags & SPEC_ACCEPT)) { j = i; break; }
        int invalid = tok_bad ? 1 : 0;
        for (int i = 0; i <= j; ++i)
            if (s_rec[i].flags & SPEC_BAD) invalid = 1;
        s_int[1] = j;
        s_int[2] = invalid;
        s_int[3] = -1;
    }
    __syncthreads();
    const int j = s_int[1];
    const bool invalid = s_int[2] != 0;
    if (!invalid && !greedy && warp == 0) {
        // the draw at j: chunk -> tile -> lane -> element, from the published sums
        const SpecRec& rj = s_rec[j];
        const float* zbase = s_z + (size_t)j * G * 2;
        int set = 0;
        float z = lane < G ? zbase[lane * 2 + 0] : 0.f;
        float incl = z;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float nb = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += nb;
        }
        float Z = __shfl_sync(0xffffffffu, incl, 31);
        if (!(Z > 0.f) && j < K) {  // the residual has no mass: draw from p_j
            set = 1;
            z = lane < G ? zbase[lane * 2 + 1] : 0.f;
            incl = z;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float nb = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += nb;
            }
            Z = __shfl_sync(0xffffffffu, incl, 31);
        }
        const float t = rj.u * Z;
        const unsigned hit = __ballot_sync(0xffffffffu, lane < G && incl > t);
        const unsigned nz = __ballot_sync(0xffffffffu, lane < G && z > 0.f);
        const int owner = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : 0);
        bool last_mode = hit == 0;
        const float t_loc = t - __shfl_sync(0xffffffffu, incl - z, owner);
        int olo, ohi;
        chunk_range(V, owner, G, olo, ohi);
        const int ntiles = (ohi - olo + TILE - 1) / TILE;
        const float* ts = reinterpret_cast<const float*>(A.ws + A.wl.tile_off) +
                          ((((size_t)b * (K + 1) + j) * G + owner) * 2 + set) * A.wl.ntiles;
        int tile = -1, last_nz_tile = -1;
        float t_tile = 0.f, cum = 0.f;
        for (int base = 0; base < ntiles && tile < 0; base += 32) {
            const float v = (base + lane < ntiles) ? __ldcg(&ts[base + lane]) : 0.f;
            float in = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float nb = __shfl_up_sync(0xffffffffu, in, o);
                if (lane >= o) in += nb;
            }
            const unsigned nzb = __ballot_sync(0xffffffffu, v > 0.f);
            if (nzb) last_nz_tile = base + 31 - __clz(nzb);
            const unsigned h = last_mode ? 0u : __ballot_sync(0xffffffffu, cum + in > t_loc);
            if (h) {
                const int f = __ffs(h) - 1;
                tile = base + f;
                t_tile = t_loc - (cum + __shfl_sync(0xffffffffu, in - v, f));
            }
            cum += __shfl_sync(0xffffffffu, in, 31);
        }
        if (tile < 0) {
            tile = last_nz_tile;
            last_mode = true;
        }
        int token = -1;
        if (tile >= 0) {
            const int e0 = olo + tile * TILE + lane * VEC;
            const unsigned char* trow = reinterpret_cast<const unsigned char*>(a.target) + ((size_t)b * (K + 1) + j) * V * tsz;
            float l[VEC], d[VEC], wr[VEC], wp[VEC];
            load8<TDT>(trow, e0, ohi, true, neg_inf(), l);
            if (j < K) {
                const unsigned char* drow = reinterpret_cast<const unsigned char*>(a.draft) + ((size_t)b * K + j) * V * dsz;
                load8<DDT>(drow, e0, ohi, true, DK == DK_LOGITS ? neg_inf() : 0.f, d);
            } else {
#pragma unroll
                for (int q = 0; q < VEC; ++q) d[q] = DK == DK_LOGITS ? neg_inf() : 0.f;
            }
            const float c = LOG2E / a.temperature[b];
            const float inv_sd = (DK == DK_LOGITS && j < K) ? 1.f / rj.ds : 0.f;
            spec_weights8<DK>(l, d, c, rj.tm, 1.f / rj.ts, rj.dm, inv_sd, wr, wp);
            float w[VEC];
#pragma unroll
            for (int q = 0; q < VEC; ++q) w[q] = (set == 0 && j < K) ? wr[q] : wp[q];
            float ls = 0.f;
#pragma unroll
            for (int q = 0; q < VEC; ++q) ls += w[q];
            float in = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float nb = __shfl_up_sync(0xffffffffu, in, o);
                if (lane >= o) in += nb;
            }
            const unsigned h = last_mode ? 0u : __ballot_sync(0xffffffffu, in > t_tile);
            const unsigned nzl = __ballot_sync(0xffffffffu, ls > 0.f);
            int f;
            bool lane_last = last_mode;
            if (h) {
                f = __ffs(h) - 1;
            } else {
                f = nzl ? 31 - __clz(nzl) : 0;
                lane_last = true;
            }
            const float t_lane = t_tile - __shfl_sync(0xffffffffu, in - ls, f);
            if (lane == f) {
                int pick = -1, last_nz = -1;
                float run = 0.f;
#pragma unroll
                for (int q = 0; q < VEC; ++q) {
                    if (w[q] > 0.f) last_nz = q;
                    run += w[q];
                    if (!lane_last && pick < 0 && run > t_lane) pick = q;
                }
                if (pick < 0) pick = last_nz < 0 ? 0 : last_nz;
                token = e0 + pick;
            }
            token = __shfl_sync(0xffffffffu, token, f);
        }
        if (lane == 0) s_int[3] = token;
    }
    __syncthreads();
    const int final_tok = greedy ? s_rec[j].argmax : s_int[3];
    int32_t* ot = a.out_tokens + (size_t)b * (K + 1);
    for (int i = threadIdx.x; i <= K; i += NT)
        ot[i] = invalid ? -1 : (i < j ? s_tok[i] : (i == j ? final_tok : -1));
    if (a.out_accept_prob)
        for (int i = threadIdx.x; i < K; i += NT) {
            float ap = -1.f;
            if (!invalid && i <= j) ap = greedy ? ((s_rec[i].flags & SPEC_ACCEPT) ? 1.f : 0.f) : fminf(s_rec[i].ratio, 1.f);
            a.out_accept_prob[(size_t)b * K + i] = ap;
        }
    if (threadIdx.x == 0) {
        a.out_count[b] = invalid ? 0 : j + 1;
        unsigned* counter = reinterpret_cast<unsigned*>(A.ws + A.wl.counter_off) + b;
        *counter = 0u;  // ready for the next call on this workspace
    }
}


size_t spec_workspace_bytes(int B, int K, int V, int G) { return spec_ws_layout(B, K, V, G).total; }

size_t spec_smem_bytes(int V, int K, int G, int tsz, int dsz, int* t_bytes, int* d_bytes, int* fin_off) {
    const size_t nvec = (size_t)(V + VEC - 1) / VEC, cmax = ((nvec + G - 1) / G) * VEC;
    const size_t tb = (cmax * tsz + 15) & ~(size_t)15, db = (cmax * dsz + 15) & ~(size_t)15;
    const size_t ntiles = (cmax + TILE - 1) / TILE;
    const size_t fin = STAGE_HEADER + tb + db + ((2 * ntiles * sizeof(float) + 15) & ~(size_t)15);
    if (t_bytes) *t_bytes = (int)tb;
    if (d_bytes) *d_bytes = (int)db;
    if (fin_off) *fin_off = (int)fin;
    return fin + (size_t)(K + 1) * G * 2 * sizeof(float);
}

template <int TDT, int DDT, int DK>
static cudaError_t launch_chain_spec_t(const ChainArgs& a, void* ws, int G, cudaStream_t stream) {
    auto kern = chain_spec_kernel<TDT, DDT, DK>;
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
    SpecArgs A;
    A.a = a;
    A.ws = reinterpret_cast<unsigned char*>(ws);
    A.wl = spec_ws_layout(a.B, a.K, a.V, G);
    const size_t smem = spec_smem_bytes(a.V, a.K, G, TDT == DT_BF16 ? 2 : 4, DDT == DT_BF16 ? 2 : 4, &A.t_bytes,
                                        &A.d_bytes, &A.fin_off);
    if (smem > (size_t)max_dyn) return cudaErrorInvalidClusterSize;  // caller takes another kernel
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
    cfg.gridDim = dim3((unsigned)G, (unsigned)(a.K + 1), (unsigned)a.B);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
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
