// sv_stage.cuh -- shared-memory staging of a CTA's chunk of vocabulary rows.
//
// A CTA owns elements [lo, hi) of each row it works on.  The chunk is brought
// into shared memory with one 1-D bulk copy per row (cp.async.bulk, completion
// counted on an mbarrier), so the softmax statistics, the acceptance test and
// the replacement draw all read shared memory and a row crosses HBM once.
// Waits on the mbarrier are bounded: a copy that never lands is reported as a
// failed wait (the row is then marked invalid) instead of hanging the kernel.
// Staging requires 16-byte aligned rows; other rows take the register-streaming
// path of sv_common.cuh.
#pragma once

#include "sv_common.cuh"

namespace sv {

// Elements per 16-byte smem vector step: 8 values (bf16: one 16 B read; fp32: two).
template <int DT>
__device__ __forceinline__ void smem_load8(const unsigned char* buf, int e, int n, float pad, float x[VEC]) {
    if (e + VEC <= n) {
        if (DT == DT_BF16) {
            const uint4 v = *reinterpret_cast<const uint4*>(buf + (size_t)e * 2);
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
            x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
        } else {
            const float4 a = *reinterpret_cast<const float4*>(buf + (size_t)e * 4);
            const float4 b = *reinterpret_cast<const float4*>(buf + (size_t)e * 4 + 16);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            if (e + j < n) {
                x[j] = (DT == DT_BF16)
                           ? __uint_as_float((uint32_t)(reinterpret_cast<const unsigned short*>(buf))[e + j] << 16)
                           : reinterpret_cast<const float*>(buf)[e + j];
            } else {
                x[j] = pad;
            }
        }
    }
}

// Eight staged elements e..e+7, all below the chunk's end (no bounds test).
template <int DT>
__device__ __forceinline__ void smem_load8_full(const unsigned char* buf, int e, float x[VEC]) {
    if (DT == DT_BF16) {
        const uint4 v = *reinterpret_cast<const uint4*>(buf + (size_t)e * 2);
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    } else {
        const float4 a = *reinterpret_cast<const float4*>(buf + (size_t)e * 4);
        const float4 b = *reinterpret_cast<const float4*>(buf + (size_t)e * 4 + 16);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
}

template <int DT>
__device__ __forceinline__ float smem_elem(const unsigned char* buf, int e) {
    return (DT == DT_BF16) ? __uint_as_float((uint32_t)(reinterpret_cast<const unsigned short*>(buf))[e] << 16)
                           : reinterpret_cast<const float*>(buf)[e];
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Maximum of one thread's share of the n staged elements (NaN propagates).  bf16 rows
// are scanned as packed pairs: three max.bf16x2 per 16-byte vector, no unpacking.
template <int DT>
__device__ __forceinline__ float smem_thread_max(const unsigned char* buf, int n) {
    if (DT == DT_BF16) {
        uint32_t acc = 0xff80ff80u;  // (-inf, -inf)
        int e = (int)threadIdx.x * VEC;
        for (; e + VEC <= n; e += NT * VEC) {
            const uint4 v = *reinterpret_cast<const uint4*>(buf + (size_t)e * 2);
            acc = bmax2_nan(acc, bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w)));
        }
        float m = fmax_nan(bf16_lo(acc), bf16_hi(acc));
        if (e < n) {  // a partial last vector
            float x[VEC];
            smem_load8<DT>(buf, e, n, neg_inf(), x);
            m = fmax_nan(m, vmax8(x));
        }
        return m;
    }
    float m = neg_inf();
    for (int e = (int)threadIdx.x * VEC; e < n; e += NT * VEC) {
        float x[VEC];
        smem_load8<DT>(buf, e, n, neg_inf(), x);
        m = fmax_nan(m, vmax8(x));
    }
    return m;
}

// (max, sum 2^((l - max) c)) of one thread's share of the n staged elements, in two
// passes over shared memory: the maximum first, then independent exponentials with
// no rescaling, each argument a single FFMA l*c - max*c.
template <int DT>
__device__ __forceinline__ LSE smem_thread_lse(const unsigned char* buf, int n, float c) {
    const float m = smem_thread_max<DT>(buf, n);
    LSE acc{m, 0.f, m != m ? 1 : 0};
    if (!(m > neg_inf()) || acc.bad) return acc;
    const float mc = m * c;
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
    int e = (int)threadIdx.x * VEC;
    for (; e + NT * VEC + VEC <= n; e += 2 * NT * VEC) {  // two full vectors per iteration
        float x[VEC], y[VEC];
        smem_load8_full<DT>(buf, e, x);
        smem_load8_full<DT>(buf, e + NT * VEC, y);
        exp2_sum8(x, c, mc, a0, a1);
        exp2_sum8(y, c, mc, a0, a1);
    }
    for (; e < n; e += NT * VEC) {  // at most one more vector, possibly ragged
        float x[VEC];
        smem_load8<DT>(buf, e, n, neg_inf(), x);
        exp2_sum8(x, c, mc, a0, a1);
    }
    acc.s = (a0.x + a0.y) + (a1.x + a1.y);
    return acc;
}

// smem_thread_lse of a target chunk and a draft-logit chunk at once: the two maxima, then
// one loop over both chunks (twice the independent exponentials per iteration, which
// helps a CTA that is alone on its SM).
template <int TDT, int DDT>
__device__ __forceinline__ void smem_thread_lse2(const unsigned char* tb, const unsigned char* db, int n, float c,
                                                 LSE& t, LSE& d) {
    const float mt = smem_thread_max<TDT>(tb, n), md = smem_thread_max<DDT>(db, n);
    t = LSE{mt, 0.f, mt != mt ? 1 : 0};
    d = LSE{md, 0.f, md != md ? 1 : 0};
    const bool use_t = mt > neg_inf() && !t.bad, use_d = md > neg_inf() && !d.bad;
    if (!use_t || !use_d) {  // a degenerate chunk: the single-row loops
        if (use_t) t = smem_thread_lse<TDT>(tb, n, c);
        if (use_d) d = smem_thread_lse<DDT>(db, n, c);
        return;
    }
    const float mtc = mt * c, mdc = md * c;
    float2 t0 = make_float2(0.f, 0.f), t1 = t0, d0 = t0, d1 = t0;
    for (int e = (int)threadIdx.x * VEC; e < n; e += NT * VEC) {
        float x[VEC], y[VEC];
        smem_load8<TDT>(tb, e, n, neg_inf(), x);
        smem_load8<DDT>(db, e, n, neg_inf(), y);
        exp2_sum8(x, c, mtc, t0, t1);
        exp2_sum8(y, c, mdc, d0, d1);
    }
    t.s = (t0.x + t0.y) + (t1.x + t1.y);
    d.s = (d0.x + d0.y) + (d1.x + d1.y);
}

// One 16-byte vector of a bf16 row in global memory at e (e a multiple of 8): elements
// at or beyond hi read as -inf.
__device__ __forceinline__ uint4 ld_bf16x8_ragged(const unsigned short* r, int e, int hi) {
    if (e + VEC <= hi) return ld_nc_v4(r + e);
    uint32_t w[4] = {0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u};
    for (int j = 0; j < VEC && e + j < hi; ++j) {
        const uint32_t h = (uint32_t)__ldg(r + e + j);
        w[j >> 1] = (j & 1) ? ((w[j >> 1] & 0x0000ffffu) | (h << 16)) : ((w[j >> 1] & 0xffff0000u) | h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Online (max, sum) update with a block of values whose maximum is vm: the running sum is
// rescaled only when the maximum grows; a NaN maximum marks the partial invalid.
__device__ __forceinline__ bool lse_online_max(LSE& acc, float& mc, float vm, float c, float2& a0, float2& a1) {
    if (vm != vm) acc.bad = BAD_DATA;
    if (vm > acc.m) {
        const float f = ex2((acc.m - vm) * c);
        a0 = fmul2(a0, make_float2(f, f));
        a1 = fmul2(a1, make_float2(f, f));
        acc.m = vm;
        mc = vm * c;
    }
    return acc.m > neg_inf();
}

__device__ __forceinline__ void exp2_sum_bf16x8(const uint4& v, float c, float mc, float2& a0, float2& a1) {
    const float x[VEC] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                          bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    exp2_sum8(x, c, mc, a0, a1);
}

// (max, sum 2^((l - max) c)) of one thread's share of elements [lo, hi) of a row in global
// memory (16-byte aligned; lo a multiple of 8), online.  bf16 rows: the thread's vectors in
// groups of five, all five loads in flight at once and kept packed until used; one maximum
// per group (max.bf16x2, no unpacking) and one rescale test per group, then the
// exponentials.  Vectors at or beyond hi read as -inf and are skipped.  A CTA's share of a
// 152064-element row split eight ways is 9 or 10 vectors per thread: two groups.
template <int DT>
__device__ __forceinline__ LSE global_thread_lse(const void* row, int lo, int hi, float c) {
    if (DT != DT_BF16) return thread_lse<DT, 2>(row, lo, hi, true, c);
    constexpr int U = 5, STEP = NT * VEC;
    LSE acc{neg_inf(), 0.f, 0};
    float mc = 0.f;
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
    for (int e0 = lo + (int)threadIdx.x * VEC; e0 < hi; e0 += U * STEP) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * STEP;
            v[u] = e + VEC <= hi ? ld_nc_v4(r + e)
                                 : (e < hi ? ld_bf16x8_ragged(r, e, hi)
                                           : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u));
        }
        uint32_t pm = bmax2_nan(bmax2_nan(v[0].x, v[0].y), bmax2_nan(v[0].z, v[0].w));
#pragma unroll
        for (int u = 1; u < U; ++u) pm = bmax2_nan(pm, bmax2_nan(bmax2_nan(v[u].x, v[u].y), bmax2_nan(v[u].z, v[u].w)));
        if (lse_online_max(acc, mc, fmax_nan(bf16_lo(pm), bf16_hi(pm)), c, a0, a1)) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (e0 + u * STEP < hi) exp2_sum_bf16x8(v[u], c, mc, a0, a1);
        }
    }
    acc.s = (a0.x + a0.y) + (a1.x + a1.y);
    return acc;
}

// argmax (lowest index on ties) of the n staged elements; indices reported as lo + local.
template <int DT>
__device__ __forceinline__ ArgMax smem_thread_argmax(const unsigned char* buf, int n, int lo) {
    ArgMax acc{neg_inf(), 0x7fffffff, 0};
    for (int e = (int)threadIdx.x * VEC; e < n; e += NT * VEC) {
        float x[VEC];
        smem_load8<DT>(buf, e, n, neg_inf(), x);
        const float vm = vmax8(x);
        if (vm != vm) acc.bad = 1;
        if (vm > acc.v) {
            int j = 0;
#pragma unroll
            for (int t = VEC - 1; t >= 0; --t)
                if (x[t] == vm) j = t;
            acc.v = vm;
            acc.i = lo + e + j;
        }
    }
    return acc;
}

// The sum slot of a pushed (max, sum) partial: the sum, or a NaN whose payload names
// the flag (a timeout takes precedence over invalid data).
__device__ __forceinline__ float flagged_sum(const LSE& s) {
    if (s.bad & BAD_TIMEOUT) return __uint_as_float(NAN_TIMEOUT);
    if (s.bad) return __uint_as_float(NAN_BAD_DATA);
    return s.s;
}

// Flags of a received sum slot (0 for a number).
__device__ __forceinline__ int sum_flags(float v) {
    if (v == v) return 0;
    return __float_as_uint(v) == NAN_TIMEOUT ? BAD_TIMEOUT : BAD_DATA;
}

__device__ __forceinline__ bool row_bad_s(const LSE& s) {
    return s.bad || !(s.m > neg_inf()) || s.m == pos_inf();
}

// Cluster combine of a position's statistics: two (max, sum) pairs, plus two values
// gathered at the drafted token by whichever CTA owns it (has = 1 in exactly one CTA).
struct PosStats {
    LSE t, d;
    float tx, dx;
    int found;
};

// TWO: a draft row takes part (draft logits); otherwise only the target pair is reduced.
template <bool TWO>
__device__ __forceinline__ PosStats cluster_pos_stats(LSE t, LSE d, float c, float tx, float dx, int has,
                                                      BlockScratch& sc, int& phase) {
    // Lanes 0..G-1 of every warp send the warp's partials into CTA `lane`'s inbox;
    // warp 0 also sends the values thread 0 gathered at x_k.  Each CTA waits for its
    // own inbox (its barrier counts the bytes) and combines from local memory: every
    // lane takes up to four partials, then a warp maximum, one rescale per partial and
    // a warp sum.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = (int)cluster_size(), me = (int)cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, (uint32_t)(G * (NW + 1)) * 16u);
    if (TWO) {
        lse2_warp_reduce(t, d, c);
    } else {
        lse_warp_reduce(t, c);
    }
    if (lane < G) {
        const float4 v = make_float4(t.m, flagged_sum(t), TWO ? d.m : neg_inf(), TWO ? flagged_sum(d) : 0.f);
        st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][warp], (uint32_t)lane), v, xchg_bar(sc, phase, lane));
    }
    if (warp == 0) {
        const float gtx = __shfl_sync(0xffffffffu, tx, 0), gdx = __shfl_sync(0xffffffffu, dx, 0);
        const int ghas = __shfl_sync(0xffffffffu, has, 0);
        if (lane < G)
            st_async_v4(dsmem_addr(&sc.inbox.gath[buf][me], (uint32_t)lane), make_float4(gtx, gdx, (float)ghas, 0.f),
                        xchg_bar(sc, phase, lane));
    }
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        const int E = G * NW;  // at most 16 * 8 = 128 partials: four per lane
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? sc.inbox.part[buf][e / NW][e % NW] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
        }
        float Mt = neg_inf(), Md = neg_inf();
        int bt = 0, bd = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Mt = fmaxf(Mt, v[i].x);
            Md = fmaxf(Md, v[i].z);
            bt |= sum_flags(v[i].y);
            bd |= sum_flags(v[i].w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
            if (TWO) Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, o));
        }
        float St = 0.f, Sd = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (v[i].x > neg_inf() && v[i].y == v[i].y) St += v[i].y * ex2((v[i].x - Mt) * c);
            if (TWO && v[i].z > neg_inf() && v[i].w == v[i].w) Sd += v[i].w * ex2((v[i].z - Md) * c);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            St += __shfl_xor_sync(0xffffffffu, St, o);
            if (TWO) Sd += __shfl_xor_sync(0xffffffffu, Sd, o);
        }
        // a wait that gave up voids the row (and is reported as a timeout)
        bt = (int)__reduce_or_sync(0xffffffffu, (unsigned)bt) | (ok ? 0 : BAD_TIMEOUT);
        bd = (int)__reduce_or_sync(0xffffffffu, (unsigned)bd) | (ok ? 0 : BAD_TIMEOUT);
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < G) gv = sc.inbox.gath[buf][lane];
        const unsigned owners = __ballot_sync(0xffffffffu, gv.z != 0.f);
        const int src = owners ? __ffs(owners) - 1 : 0;
        const float gx = __shfl_sync(0xffffffffu, gv.x, src), gd = __shfl_sync(0xffffffffu, gv.y, src);
        if (lane == 0) {
            sc.bf[0] = Mt; sc.bf[1] = St; sc.bf[2] = TWO ? Md : neg_inf(); sc.bf[3] = TWO ? Sd : 0.f;
            sc.bf[4] = gx; sc.bf[5] = gd;
            sc.bi[0] = bt; sc.bi[1] = TWO ? bd : 0; sc.bi[2] = owners ? 1 : 0;
        }
    }
    __syncthreads();
    PosStats r;
    r.t = LSE{sc.bf[0], sc.bf[1], sc.bi[0]};
    r.d = LSE{sc.bf[2], sc.bf[3], sc.bi[1]};
    r.tx = sc.bf[4];
    r.dx = sc.bf[5];
    r.found = sc.bi[2];
    ++phase;
    return r;
}

// Weight functors over staged chunks (row coordinates e0 >= lo; elements >= hi weigh 0).
template <int TDT>
struct StagedP {  // w = p = 2^((l - m) c) / S
    const unsigned char* tb;
    int lo;
    float c, m, inv_s;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC];
        smem_load8<TDT>(tb, e0 - lo, hi - lo, neg_inf(), l);
        exp2_scale8(l, c, m * c, inv_s, w);
    }
    __device__ __forceinline__ void eval8_full(int e0, float w[VEC]) const {
        float l[VEC];
        smem_load8_full<TDT>(tb, e0 - lo, l);
        exp2_scale8(l, c, m * c, inv_s, w);
    }
};

// w_j = max(0, p_j - q_j) from eight probabilities of each (exact subtraction, no contraction).
__device__ __forceinline__ void residual8(const float p[VEC], const float q[VEC], float w[VEC]) {
#pragma unroll
    for (int j = 0; j < VEC; j += 2) {
        const float2 r = fsub2(make_float2(p[j], p[j + 1]), make_float2(q[j], q[j + 1]));
        w[j] = fmaxf(r.x, 0.f);
        w[j + 1] = fmaxf(r.y, 0.f);
    }
}

// Residual weights with the target chunk staged and the draft-logit row read from global
// memory (it was streamed for its statistics just before, so from L2).  The draw needs
// the weights only up to a common factor, so they are S_t * max(0, p - q) =
// max(0, e_t - rho e_d), with e = 2^((l - M) c) and rho = S_t / S_d: one multiply per
// element fewer than normalising both rows.  Where the two rows and their statistics are
// equal, rho is exactly 1 and every weight exactly 0, as for p - q.
template <int TDT, int DDT>
struct StagedResidualD {
    static constexpr int kTilesInFlight = 4;  // global loads: several tiles in flight per warp
    const unsigned char* tb;
    const void* drow;
    int lo;
    float c, mt, md, rho;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC], d[VEC];
        smem_load8<TDT>(tb, e0 - lo, hi - lo, neg_inf(), l);
        load8<DDT>(drow, e0, hi, true, neg_inf(), d);
        weights(l, d, w);
    }
    __device__ __forceinline__ void eval8_full(int e0, float w[VEC]) const {
        float l[VEC], d[VEC];
        smem_load8_full<TDT>(tb, e0 - lo, l);
        load8<DDT>(drow, e0, e0 + VEC, true, neg_inf(), d);
        weights(l, d, w);
    }
    __device__ __forceinline__ void weights(float l[VEC], const float d[VEC], float w[VEC]) const {
        float q[VEC];
        const float2 cc = make_float2(c, c), mt2 = make_float2(-mt * c, -mt * c), md2 = make_float2(-md * c, -md * c);
        const float2 rr = make_float2(rho, rho);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
            const float2 yt = ffma2(make_float2(l[j], l[j + 1]), cc, mt2);
            const float2 yd = ffma2(make_float2(d[j], d[j + 1]), cc, md2);
            const float2 qd = fmul2(make_float2(ex2(yd.x), ex2(yd.y)), rr);
            l[j] = ex2(yt.x);
            l[j + 1] = ex2(yt.y);
            q[j] = qd.x;
            q[j + 1] = qd.y;
        }
        residual8(l, q, w);
    }
};

template <int TDT, int DDT, int DK>
struct StagedResidual {  // w = max(0, p - q)
    const unsigned char* tb;
    const unsigned char* db;
    int lo;
    float c, mt, inv_st, md, inv_sd;
    __device__ __forceinline__ void eval8(int e0, int hi, float w[VEC]) const {
        float l[VEC], d[VEC];
        smem_load8<TDT>(tb, e0 - lo, hi - lo, neg_inf(), l);
        smem_load8<DDT>(db, e0 - lo, hi - lo, DK == DK_LOGITS ? neg_inf() : 0.f, d);
        weights(l, d, w);
    }
    __device__ __forceinline__ void eval8_full(int e0, float w[VEC]) const {
        float l[VEC], d[VEC];
        smem_load8_full<TDT>(tb, e0 - lo, l);
        smem_load8_full<DDT>(db, e0 - lo, d);
        weights(l, d, w);
    }
    __device__ __forceinline__ void weights(const float l[VEC], const float d[VEC], float w[VEC]) const {
        float p[VEC];
        exp2_scale8(l, c, mt * c, inv_st, p);
        if (DK == DK_LOGITS) {
            float q[VEC];
            exp2_scale8(d, c, md * c, inv_sd, q);
            residual8(p, q, w);
        } else {
            residual8(p, d, w);
        }
    }
};

}  // namespace sv
