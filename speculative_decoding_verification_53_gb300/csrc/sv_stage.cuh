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

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Order this CTA's generic-proxy accesses of shared memory before later async-proxy writes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after a bounded number
// of polls (about a quarter of a second) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 32) __nanosleep(64);
    }
    return false;
}

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

template <int DT>
__device__ __forceinline__ float smem_elem(const unsigned char* buf, int e) {
    return (DT == DT_BF16) ? __uint_as_float((uint32_t)(reinterpret_cast<const unsigned short*>(buf))[e] << 16)
                           : reinterpret_cast<const float*>(buf)[e];
}

// Online (max, sum 2^((l - max) c)) of the n staged elements, one thread's share.
template <int DT>
__device__ __forceinline__ LSE smem_thread_lse(const unsigned char* buf, int n, float c) {
    LSE acc{neg_inf(), 0.f, 0};
    for (int e = (int)threadIdx.x * VEC; e < n; e += NT * VEC) {
        float x[VEC];
        smem_load8<DT>(buf, e, n, neg_inf(), x);
        const float vm = vmax8(x);
        if (vm != vm) acc.bad = 1;
        if (vm > acc.m) {
            acc.s *= ex2((acc.m - vm) * c);
            acc.m = vm;
        }
        if (acc.m > neg_inf()) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < VEC; j += 2) {
                s0 += ex2((x[j] - acc.m) * c);
                s1 += ex2((x[j + 1] - acc.m) * c);
            }
            acc.s += s0 + s1;
        }
    }
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

__device__ __forceinline__ PosStats cluster_pos_stats(LSE t, LSE d, float c, float tx, float dx, int has,
                                                      BlockScratch& sc, int& phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    lse_warp_reduce(t, c);
    lse_warp_reduce(d, c);
    if (lane == 0) {
        sc.rf[warp][0] = t.m; sc.rf[warp][1] = t.s;
        sc.rf[warp][2] = d.m; sc.rf[warp][3] = d.s;
        sc.ri[warp][0] = t.bad; sc.ri[warp][1] = d.bad;
    }
    __syncthreads();
    Xchg& slot = sc.xchg[phase & 1];
    if (warp == 0) {
        LSE x{neg_inf(), 0.f, 0}, y{neg_inf(), 0.f, 0};
        if (lane < NW) {
            x = LSE{sc.rf[lane][0], sc.rf[lane][1], sc.ri[lane][0]};
            y = LSE{sc.rf[lane][2], sc.rf[lane][3], sc.ri[lane][1]};
        }
        lse_warp_reduce(x, c);
        lse_warp_reduce(y, c);
        if (lane == 0) {
            slot.f[0] = x.m; slot.f[1] = x.s; slot.f[2] = y.m; slot.f[3] = y.s;
            slot.f[4] = tx; slot.f[5] = dx;
            slot.i[0] = x.bad; slot.i[1] = y.bad; slot.i[2] = has;
        }
    }
    cluster_sync_all();
    if (warp == 0) {
        const uint32_t G = cluster_size();
        LSE x{neg_inf(), 0.f, 0}, y{neg_inf(), 0.f, 0};
        float gx = 0.f, gd = 0.f;
        int h = 0;
        if ((uint32_t)lane < G) {
            x.m = dsmem_ld_f32(dsmem_addr(&slot.f[0], lane));
            x.s = dsmem_ld_f32(dsmem_addr(&slot.f[1], lane));
            y.m = dsmem_ld_f32(dsmem_addr(&slot.f[2], lane));
            y.s = dsmem_ld_f32(dsmem_addr(&slot.f[3], lane));
            gx = dsmem_ld_f32(dsmem_addr(&slot.f[4], lane));
            gd = dsmem_ld_f32(dsmem_addr(&slot.f[5], lane));
            x.bad = dsmem_ld_s32(dsmem_addr(&slot.i[0], lane));
            y.bad = dsmem_ld_s32(dsmem_addr(&slot.i[1], lane));
            h = dsmem_ld_s32(dsmem_addr(&slot.i[2], lane));
        }
        lse_warp_reduce(x, c);
        lse_warp_reduce(y, c);
        const unsigned owners = __ballot_sync(0xffffffffu, h != 0);
        const int src = owners ? __ffs(owners) - 1 : 0;
        gx = __shfl_sync(0xffffffffu, gx, src);
        gd = __shfl_sync(0xffffffffu, gd, src);
        if (lane == 0) {
            sc.bf[0] = x.m; sc.bf[1] = x.s; sc.bf[2] = y.m; sc.bf[3] = y.s;
            sc.bf[4] = gx; sc.bf[5] = gd;
            sc.bi[0] = x.bad; sc.bi[1] = y.bad; sc.bi[2] = owners ? 1 : 0;
        }
    }
    __syncthreads();
    PosStats r;
    r.t = LSE{sc.bf[0], sc.bf[1], sc.bi[0]};
    r.d = LSE{sc.bf[2], sc.bf[3], sc.bi[1]};
    r.tx = sc.bf[4];
    r.dx = sc.bf[5];
    r.found = sc.bi[2];
    __syncthreads();
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
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[j] = ex2((l[j] - m) * c) * inv_s;
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
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float p = ex2((l[j] - mt) * c) * inv_st;
            const float q = (DK == DK_LOGITS) ? ex2((d[j] - md) * c) * inv_sd : d[j];
            w[j] = fmaxf(p - q, 0.f);
        }
    }
};

}  // namespace sv
