// sv_common.cuh -- device building blocks of the verify kernels (sm_103a).
//
// Row statistics for the temperature softmax (online max and sum of exp2),
// argmax with lowest-index ties, Philox4x64-10 uniforms, thread-block-cluster
// exchange through distributed shared memory, and the inverse-CDF draw over a
// vocabulary row that is split across the CTAs of a cluster.
//
// The rule these implement is the accept/reject step of speculative decoding
// ("[논문 리뷰] Fast Inference from Transformers via Speculative Decoding",
// section 2; "Speculative Decoding and EAGLE", section "정확성 규칙").
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int NT = 256;            // threads per CTA
constexpr int NW = NT / 32;        // warps per CTA
constexpr int VEC = 8;             // elements per vector step (16 B of bf16, 32 B of fp32)
constexpr int TILE = 32 * VEC;     // elements per draw tile (one warp, 8 per lane)
constexpr int UNROLL = 4;          // vector steps in flight per thread
constexpr int MAX_K = 64;          // chain drafts per row
constexpr int MAX_NODES = 1024;    // tree nodes per row
constexpr int MAX_CLUSTER = 16;
constexpr float LOG2E = 1.4426950408889634f;

enum DTypeCode { DT_F32 = 0, DT_BF16 = 1 };
enum DraftCode { DK_PROBS = 0, DK_LOGITS = 1 };

// ------------------------------------------------------------------ math

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes per instruction (Blackwell's packed f32x2 arithmetic).  Each lane is
// rounded exactly as the scalar instruction would round it; the exponential loops use
// these to halve their FMA and add instructions (they are issue-bound, not exp-bound).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Sum of eight values, pairwise on the packed two-lane adder.
__device__ __forceinline__ float sum8(const float w[8]) {
    const float2 a = fadd2(make_float2(w[0], w[1]), make_float2(w[2], w[3]));
    const float2 b = fadd2(make_float2(w[4], w[5]), make_float2(w[6], w[7]));
    const float2 t = fadd2(a, b);
    return t.x + t.y;
}

// Sum of 2^(x_j c - mc) over eight values, as two packed accumulators.
__device__ __forceinline__ void exp2_sum8(const float x[8], float c, float mc, float2& a0, float2& a1) {
    const float2 cc = make_float2(c, c), mm = make_float2(-mc, -mc);
    const float2 y0 = ffma2(make_float2(x[0], x[1]), cc, mm), y1 = ffma2(make_float2(x[2], x[3]), cc, mm);
    const float2 y2 = ffma2(make_float2(x[4], x[5]), cc, mm), y3 = ffma2(make_float2(x[6], x[7]), cc, mm);
    a0 = fadd2(a0, fadd2(make_float2(ex2(y0.x), ex2(y0.y)), make_float2(ex2(y1.x), ex2(y1.y))));
    a1 = fadd2(a1, fadd2(make_float2(ex2(y2.x), ex2(y2.y)), make_float2(ex2(y3.x), ex2(y3.y))));
}

// Eight probabilities 2^(x_j c - mc) * inv_s.
__device__ __forceinline__ void exp2_scale8(const float x[8], float c, float mc, float inv_s, float w[8]) {
    const float2 cc = make_float2(c, c), mm = make_float2(-mc, -mc), ss = make_float2(inv_s, inv_s);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const float2 y = ffma2(make_float2(x[j], x[j + 1]), cc, mm);
        const float2 p = fmul2(make_float2(ex2(y.x), ex2(y.y)), ss);
        w[j] = p.x;
        w[j + 1] = p.y;
    }
}

// Maximum that propagates NaN (a NaN anywhere in a row must mark the row invalid).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

// ---------------------------------------------------------------- Philox

// Philox4x64 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11).  Per round the
// counter words 0 and 2 are multiplied by the two round constants, the 128-bit
// products are split, crossed with words 1 and 3 and the key; the key advances
// by the two Weyl increments between rounds.
__device__ __forceinline__ void philox4x64_10(uint64_t& x0, uint64_t& x1, uint64_t& x2, uint64_t& x3,
                                              uint64_t k0, uint64_t k1) {
    const uint64_t ma = 0xD2E7470EE14C6C93ull, mb = 0xCA5A826395121157ull;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t hi_a = __umul64hi(ma, x0), lo_a = ma * x0;
        const uint64_t hi_b = __umul64hi(mb, x2), lo_b = mb * x2;
        const uint64_t y0 = hi_b ^ x1 ^ k0;
        const uint64_t y2 = hi_a ^ x3 ^ k1;
        x0 = y0;
        x1 = lo_b;
        x2 = y2;
        x3 = lo_a;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
}

// The two uniforms of one Philox slot: r from word 0 (acceptance), u from word 1 (draw),
// each (w >> 40) * 2^-24, exactly representable in fp32.
__device__ __forceinline__ void slot_uniforms(uint64_t seed, uint64_t offset, uint64_t row, uint64_t slot,
                                              float& r, float& u) {
    uint64_t x0 = slot, x1 = row, x2 = offset, x3 = 0;
    philox4x64_10(x0, x1, x2, x3, seed, 0);
    r = (float)(uint32_t)(x0 >> 40) * (1.0f / 16777216.0f);
    u = (float)(uint32_t)(x1 >> 40) * (1.0f / 16777216.0f);
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization, so it may start while the previous kernel on the
// stream (typically the one that produced the logits) is still finishing.  pdl_wait()
// blocks until that kernel has completed and its writes are visible: it precedes every
// read of an input and every write of an output or workspace.  pdl_trigger() lets the
// next such kernel on the stream start its own launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The draft-sampling uniform of a Philox slot: word 2, on the same 24-bit grid.
__device__ __forceinline__ float slot_draft_uniform(uint64_t seed, uint64_t offset, uint64_t row, uint64_t slot) {
    uint64_t x0 = slot, x1 = row, x2 = offset, x3 = 0;
    philox4x64_10(x0, x1, x2, x3, seed, 0);
    return (float)(uint32_t)(x2 >> 40) * (1.0f / 16777216.0f);
}

// ----------------------------------------------------------------- loads

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int DT>
__device__ __forceinline__ float load_one(const void* row, int i) {
    if (DT == DT_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)row + i) << 16);
    return __ldg((const float*)row + i);
}

// Eight consecutive elements e0..e0+7 of a row (e0 a multiple of 8), widened to fp32.
// Elements at or beyond `hi` read as `pad`.  `al` says the row start is 16-byte aligned.
template <int DT>
__device__ __forceinline__ void load8(const void* row, int e0, int hi, bool al, float pad, float x[VEC]) {
    if (al && e0 + VEC <= hi) {
        if (DT == DT_BF16) {
            const uint4 v = ld_nc_v4((const unsigned short*)row + e0);
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
            x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
        } else {
            const uint4 a = ld_nc_v4((const float*)row + e0);
            const uint4 b = ld_nc_v4((const float*)row + e0 + 4);
            x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
            x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
            x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
            x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) x[j] = (e0 + j < hi) ? load_one<DT>(row, e0 + j) : pad;
    }
}

__device__ __forceinline__ float vmax8(const float x[VEC]) {
    const float a = fmax_nan(fmax_nan(x[0], x[1]), fmax_nan(x[2], x[3]));
    const float b = fmax_nan(fmax_nan(x[4], x[5]), fmax_nan(x[6], x[7]));
    return fmax_nan(a, b);
}

// ------------------------------------------------------ softmax statistics

// Flags a partial result carries (bitwise or-ed through every reduction): BAD_DATA for
// invalid data (NaN seen), BAD_TIMEOUT for a bounded wait (a bulk copy or a cluster
// exchange) that gave up before completing.
constexpr int BAD_DATA = 1;
constexpr int BAD_TIMEOUT = 2;

// NaN payloads of a pushed partial sum that stands for one of those flags.
constexpr uint32_t NAN_BAD_DATA = 0x7fc00001u;
constexpr uint32_t NAN_TIMEOUT = 0x7fc00002u;

// Running (max m, sum s of 2^((l - m) * c)) of a set of logits, c = log2(e) / T.
struct LSE {
    float m, s;
    int bad;  // BAD_DATA / BAD_TIMEOUT flags
};

__device__ __forceinline__ void lse_merge(LSE& a, const LSE& b, float c) {
    a.bad |= b.bad;
    if (b.m > a.m) {
        a.s = a.s * ex2((a.m - b.m) * c) + b.s;
        a.m = b.m;
    } else if (b.m > neg_inf()) {
        a.s += b.s * ex2((b.m - a.m) * c);
    }
}

// Warp all-reduce of two (max, sum) pairs with their chains interleaved.
__device__ __forceinline__ void lse2_warp_reduce(LSE& a, LSE& b, float c) {
    float Ma = a.m, Mb = b.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Ma = fmaxf(Ma, __shfl_xor_sync(0xffffffffu, Ma, o));
        Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
    }
    float sa = (a.m > neg_inf()) ? a.s * ex2((a.m - Ma) * c) : 0.f;
    float sb = (b.m > neg_inf()) ? b.s * ex2((b.m - Mb) * c) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sb += __shfl_xor_sync(0xffffffffu, sb, o);
    }
    a.bad = (int)__reduce_or_sync(0xffffffffu, (unsigned)a.bad);
    b.bad = (int)__reduce_or_sync(0xffffffffu, (unsigned)b.bad);
    a.m = Ma;
    a.s = sa;
    b.m = Mb;
    b.s = sb;
}

__device__ __forceinline__ LSE lse_shfl_xor(const LSE& v, int mask) {
    LSE o;
    o.m = __shfl_xor_sync(0xffffffffu, v.m, mask);
    o.s = __shfl_xor_sync(0xffffffffu, v.s, mask);
    o.bad = __shfl_xor_sync(0xffffffffu, v.bad, mask);
    return o;
}

// Warp all-reduce of (max, sum) pairs: the warp maximum first (no exponentials), then
// one rescale 2^((m - M) c) per lane and a plain sum, so the dependent chain holds a
// single exp2 instead of one per shuffle step.  Every lane ends with the warp's pair.
__device__ __forceinline__ void lse_warp_reduce(LSE& v, float c) {
    float M = v.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float s = (v.m > neg_inf()) ? v.s * ex2((v.m - M) * c) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    v.bad = (int)__reduce_or_sync(0xffffffffu, (unsigned)v.bad);
    v.m = M;
    v.s = s;
}

// One thread's pass over its vector steps of elements [lo, hi) of a row (U vector steps
// in flight).
template <int DT, int U = UNROLL>
__device__ __forceinline__ LSE thread_lse(const void* row, int lo, int hi, bool al, float c) {
    LSE acc{neg_inf(), 0.f, 0};
    const int v0 = lo / VEC, v1 = (hi + VEC - 1) / VEC;
    for (int vb = v0 + (int)threadIdx.x; vb < v1; vb += NT * U) {
        float x[U][VEC];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = vb + u * NT;
            if (v < v1) load8<DT>(row, v * VEC, hi, al, neg_inf(), x[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = vb + u * NT;
            if (v >= v1) break;
            const float vm = vmax8(x[u]);
            if (vm != vm) acc.bad = BAD_DATA;
            if (vm > acc.m) {
                acc.s *= ex2((acc.m - vm) * c);
                acc.m = vm;
            }
            if (acc.m > neg_inf()) {
                float2 a0 = make_float2(0.f, 0.f), a1 = a0;
                exp2_sum8(x[u], c, acc.m * c, a0, a1);
                acc.s += (a0.x + a0.y) + (a1.x + a1.y);
            }
        }
    }
    return acc;
}

// ----------------------------------------------------------------- argmax

struct ArgMax {
    float v;
    int i;
    int bad;  // BAD_DATA / BAD_TIMEOUT flags
};

__device__ __forceinline__ void argmax_merge(ArgMax& a, const ArgMax& b) {
    a.bad |= b.bad;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) {
        a.v = b.v;
        a.i = b.i;
    }
}

__device__ __forceinline__ void argmax_warp_reduce(ArgMax& v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax w;
        w.v = __shfl_xor_sync(0xffffffffu, v.v, o);
        w.i = __shfl_xor_sync(0xffffffffu, v.i, o);
        w.bad = __shfl_xor_sync(0xffffffffu, v.bad, o);
        argmax_merge(v, w);
    }
}

template <int DT>
__device__ __forceinline__ ArgMax thread_argmax(const void* row, int lo, int hi, bool al) {
    ArgMax acc{neg_inf(), 0x7fffffff, 0};
    const int v0 = lo / VEC, v1 = (hi + VEC - 1) / VEC;
    for (int vb = v0 + (int)threadIdx.x; vb < v1; vb += NT * UNROLL) {
        float x[UNROLL][VEC];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int v = vb + u * NT;
            if (v < v1) load8<DT>(row, v * VEC, hi, al, neg_inf(), x[u]);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int v = vb + u * NT;
            if (v >= v1) break;
            const float vm = vmax8(x[u]);
            if (vm != vm) acc.bad = 1;
            if (vm > acc.v) {  // strictly greater: the earlier (lower) index keeps ties
                int j = 0;
#pragma unroll
                for (int t = VEC - 1; t >= 0; --t)
                    if (x[u][t] == vm) j = t;
                acc.v = vm;
                acc.i = v * VEC + j;
            }
        }
    }
    return acc;
}

// --------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives and waits (release/acquire on
// shared::cluster), so DSMEM writes before it are visible after it.
// ------------------------------------------------------------- mbarriers

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

// Raise the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
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

// try_wait with a suspend-time hint: the thread may be suspended in hardware (woken when
// the phase completes) for up to `ns` nanoseconds instead of returning at once, so a
// waiting warp does not spin through issue slots other warps could use.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete.  Gives up and returns false
// after limit_ns nanoseconds (global timer) or 2^22 tries, whichever comes first.
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint64_t* bar, uint32_t parity, uint32_t limit_ns) {
    const uint32_t hint = limit_ns < 1000000u ? limit_ns : 1000000u;
    if (mbar_try_wait_for(bar, parity, hint)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try_wait_for(bar, parity, hint)) return true;
        if (global_ns() - t0 > (uint64_t)limit_ns) break;
    }
    return false;
}

// The default bound of every wait: a quarter of a second.
constexpr uint32_t WAIT_LIMIT_NS = 250000000u;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    return mbar_wait_bounded_ns(bar, parity, WAIT_LIMIT_NS);
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `p` (a shared variable of this CTA) in CTA `rank`'s shared memory window.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
    uint32_t local = (uint32_t)__cvta_generic_to_shared(p), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

// Fire-and-forget store into a peer CTA's shared memory (ordered by the next
// barrier.cluster release/acquire pair).
__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

// Store into a peer CTA's shared memory whose bytes complete a transaction count on
// that CTA's mbarrier `mbar` (a shared::cluster address): the receiver learns from its
// own barrier that the data has landed, with no cluster-wide barrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t mbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(mbar)
                 : "memory");
}

__device__ __forceinline__ void st_async_v2(uint32_t addr, float2 v, uint32_t mbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(v.x), "f"(v.y), "r"(mbar)
                 : "memory");
}


// Inbox of pushed partials.  In an exchange every CTA of the cluster stores its
// partials into every CTA's inbox (its own included) with st.async, each store
// completing its bytes on the receiver's barrier of that buffer; a CTA waits on its
// own barrier only, then combines from local shared memory.  A NaN sum marks a row
// that contained NaN.  Double-buffered by exchange number: a CTA sends exchange e+1
// only after it has read exchange e, so a buffer is never overwritten while read.
struct Inbox {
    float4 part[2][MAX_CLUSTER][NW];
    float4 gath[2][MAX_CLUSTER];  // (target value, draft value, has, -) at the drafted token
    float2 zf[2][MAX_CLUSTER];    // the draw's per-CTA total weight and failure flag
};

// Shared state of a CTA used by the block- and cluster-level reductions.
struct BlockScratch {
    uint64_t xbar[2];  // one mbarrier per inbox buffer
    Inbox inbox;
    float rf[NW][4];
    int ri[NW][2];
    float bf[8];  // broadcast floats
    int bi[8];    // broadcast ints
};

// Chunk [lo, hi) of a row owned by CTA g of G: boundaries on multiples of VEC.
__device__ __forceinline__ void chunk_range(int V, int g, int G, int& lo, int& hi) {
    const int nvec = (V + VEC - 1) / VEC;
    lo = (int)(((long long)g * nvec) / G) * VEC;
    hi = (int)(((long long)(g + 1) * nvec) / G) * VEC;
    if (hi > V) hi = V;
    if (lo > V) lo = V;
}

// Sets up the inbox barriers; every thread of every CTA of the cluster calls it once,
// before the first exchange.  Its cluster barrier makes every CTA's barriers exist
// before any peer sends.  No global memory is touched (it may precede pdl_wait).
template <class SC>
__device__ __forceinline__ void xchg_init(SC& sc) {
    if (threadIdx.x == 0) {
        mbar_init(&sc.xbar[0], 1);
        mbar_init(&sc.xbar[1], 1);
        fence_mbar_init();
    }
    cluster_sync_all();
}

// xchg_init split in two so that independent start-up work (issuing the first copies,
// loading the tokens, the Philox blocks) overlaps the cluster barrier: xchg_init_arrive
// sets up this CTA's inbox barriers and arrives; xchg_ready waits for every CTA's
// arrival and must come before the first exchange.  Every thread calls each once, in
// that order, with no other cluster barrier between them.
template <class SC>
__device__ __forceinline__ void xchg_init_arrive(SC& sc) {
    if (threadIdx.x == 0) {
        mbar_init(&sc.xbar[0], 1);
        mbar_init(&sc.xbar[1], 1);
        fence_mbar_init();
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void xchg_ready() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Exchange number `phase` uses inbox buffer phase & 1, whose barrier completes its
// (phase >> 1)-th phase.  Thread 0 arms it with the bytes all G senders will deliver.
template <class SC>
__device__ __forceinline__ void xchg_arm(SC& sc, int phase, uint32_t bytes) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&sc.xbar[phase & 1], bytes);
}

// The receiver's barrier of this exchange, in CTA `peer`'s window.
template <class SC>
__device__ __forceinline__ uint32_t xchg_bar(SC& sc, int phase, uint32_t peer) {
    return dsmem_addr(&sc.xbar[phase & 1], peer);
}

// Bounded wait for this CTA's inbox of exchange `phase` to be complete.
template <class SC>
__device__ __forceinline__ bool xchg_wait(SC& sc, int phase) {
    return mbar_wait_bounded(&sc.xbar[phase & 1], (uint32_t)(phase >> 1) & 1u);
}

// Block reduce of up to two LSE pairs, then a cluster-wide combine in rank order.
// Every thread of every CTA returns the same values.  Warp 0 sends the CTA's pairs
// into every inbox, then waits for its own and combines locally.
__device__ __forceinline__ void cluster_lse2(LSE& a, LSE& b, float c, BlockScratch& sc, int& phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t G = cluster_size(), me = cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, G * 32u);
    lse_warp_reduce(a, c);
    lse_warp_reduce(b, c);
    if (lane == 0) {
        sc.rf[warp][0] = a.m; sc.rf[warp][1] = a.s;
        sc.rf[warp][2] = b.m; sc.rf[warp][3] = b.s;
        sc.ri[warp][0] = a.bad; sc.ri[warp][1] = b.bad;
    }
    __syncthreads();
    if (warp == 0) {
        LSE x{neg_inf(), 0.f, 0}, y{neg_inf(), 0.f, 0};
        if (lane < NW) {
            x = LSE{sc.rf[lane][0], sc.rf[lane][1], sc.ri[lane][0]};
            y = LSE{sc.rf[lane][2], sc.rf[lane][3], sc.ri[lane][1]};
        }
        lse_warp_reduce(x, c);
        lse_warp_reduce(y, c);
        if ((uint32_t)lane < G) {
            const uint32_t peer = (uint32_t)lane, bar = xchg_bar(sc, phase, peer);
            st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][0], peer), make_float4(x.m, x.s, y.m, y.s), bar);
            st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][1], peer),
                        make_float4(__int_as_float(x.bad), __int_as_float(y.bad), 0.f, 0.f), bar);
        }
    }
    if (warp == 0) {
        const int ok = __all_sync(0xffffffffu, xchg_wait(sc, phase)) ? 1 : 0;
        LSE x{neg_inf(), 0.f, 0}, y{neg_inf(), 0.f, 0};
        if ((uint32_t)lane < G) {
            const float4 v = sc.inbox.part[buf][lane][0], f = sc.inbox.part[buf][lane][1];
            x = LSE{v.x, v.y, __float_as_int(f.x) | (ok ? 0 : BAD_TIMEOUT)};
            y = LSE{v.z, v.w, __float_as_int(f.y) | (ok ? 0 : BAD_TIMEOUT)};
        }
        lse_warp_reduce(x, c);
        lse_warp_reduce(y, c);
        if (lane == 0) {
            sc.bf[0] = x.m; sc.bf[1] = x.s; sc.bf[2] = y.m; sc.bf[3] = y.s;
            sc.bi[0] = x.bad; sc.bi[1] = y.bad;
        }
    }
    __syncthreads();
    a = LSE{sc.bf[0], sc.bf[1], sc.bi[0]};
    b = LSE{sc.bf[2], sc.bf[3], sc.bi[1]};
    __syncthreads();
    ++phase;
}

__device__ __forceinline__ ArgMax cluster_argmax(ArgMax a, BlockScratch& sc, int& phase) {
    // Lanes 0..G-1 of every warp send the warp's (max, index, NaN flag) into CTA
    // `lane`'s inbox; each CTA waits for its own inbox and reduces locally.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = (int)cluster_size(), me = (int)cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, (uint32_t)(G * NW) * 16u);
    argmax_warp_reduce(a);
    if (lane < G)
        st_async_v4(dsmem_addr(&sc.inbox.part[buf][me][warp], (uint32_t)lane),
                    make_float4(a.v, __int_as_float(a.i), __int_as_float(a.bad), 0.f), xchg_bar(sc, phase, lane));
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        ArgMax x{neg_inf(), 0x7fffffff, ok ? 0 : BAD_TIMEOUT};
        for (int e = lane; e < G * NW; e += 32) {
            const float4 v = sc.inbox.part[buf][e / NW][e % NW];
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

// Cluster-wide sum of two floats (fixed order, identical in every CTA).  Warp 0 sends
// the CTA's pair into every inbox, waits for its own and adds it in rank order.  A
// wait that gives up returns NaN sums.
__device__ __forceinline__ float2 cluster_sum2(float2 v, BlockScratch& sc, int& phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t G = cluster_size(), me = cluster_rank();
    const int buf = phase & 1;
    xchg_arm(sc, phase, G * 8u);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    if (lane == 0) { sc.rf[warp][0] = v.x; sc.rf[warp][1] = v.y; }
    __syncthreads();
    if (warp == 0) {
        float2 x = make_float2(0.f, 0.f);
        if (lane < NW) x = make_float2(sc.rf[lane][0], sc.rf[lane][1]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            x.x += __shfl_xor_sync(0xffffffffu, x.x, o);
            x.y += __shfl_xor_sync(0xffffffffu, x.y, o);
        }
        if ((uint32_t)lane < G)
            st_async_v2(dsmem_addr(&sc.inbox.zf[buf][me], (uint32_t)lane), x, xchg_bar(sc, phase, (uint32_t)lane));
    }
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        float2 x = make_float2(0.f, 0.f);
        if ((uint32_t)lane < G) x = ok ? sc.inbox.zf[buf][lane] : make_float2(nanf(""), nanf(""));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            x.x += __shfl_xor_sync(0xffffffffu, x.x, o);
            x.y += __shfl_xor_sync(0xffffffffu, x.y, o);
        }
        if (lane == 0) { sc.bf[0] = x.x; sc.bf[1] = x.y; }
    }
    __syncthreads();
    float2 r = make_float2(sc.bf[0], sc.bf[1]);
    __syncthreads();
    ++phase;
    return r;
}

// ------------------------------------------------------------------ draw

// Inverse-CDF draw over a row split across the cluster: the token is the smallest
// index i whose prefix sum of weights exceeds u * Z (Z the row's total weight).
// The weight functor WF provides eval8(e0, hi, w[8]) for elements e0..e0+7 (0 beyond hi).
//
// Pass 1: per-tile sums (tile = 256 elements, one warp) into shared memory, CTA
// totals exchanged across the cluster.  Pass 2: the CTA whose prefix range holds
// u * Z narrows it to a tile, a lane and an element.  Where rounding leaves the
// target past the last element of a range, the last element with non-zero weight
// in that range is taken.
//
// Returns in *out_token the token (valid in the owner CTA) and the owner rank;
// returns false (no owner) when the total weight is zero.
struct DrawResult {
    int owner;
    int token;
    float Z;
    int failed;  // some CTA reported fail_in (a staging wait that gave up): the draw is void
};

// The draw given the tile sums of this CTA's chunk (tile t: elements lo + 256 t ..);
// wf evaluates the weights of the one tile the owner CTA searches.  The caller has
// synchronised the CTA after writing tile_sum.
template <class WF, class SC>
__device__ __forceinline__ DrawResult cluster_draw_from_tiles(const WF& wf, int lo, int hi, float u, const float* tile_sum,
                                              SC& sc, int& phase, int fail_in = 0) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ntiles = (hi - lo + TILE - 1) / TILE;
    xchg_arm(sc, phase, cluster_size() * 8u);
    if (warp == 0) {
        float z = 0.f;
        for (int t = lane; t < ntiles; t += 32) z += tile_sum[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const uint32_t Gp = cluster_size(), me = cluster_rank();
        if ((uint32_t)lane < Gp)  // send (total, failure) into every inbox
            st_async_v2(dsmem_addr(&sc.inbox.zf[phase & 1][me], (uint32_t)lane), make_float2(z, (float)fail_in),
                        xchg_bar(sc, phase, (uint32_t)lane));
    }
    if (warp == 0) {
        const uint32_t G = cluster_size();
        const bool ok = __all_sync(0xffffffffu, xchg_wait(sc, phase));
        float z = 0.f;
        int fl = ok ? 0 : 1;
        if ((uint32_t)lane < G) {
            const float2 v = sc.inbox.zf[phase & 1][lane];
            z = v.x;
            fl |= v.y != 0.f ? 1 : 0;
        }
        const int any_fail = __any_sync(0xffffffffu, fl != 0) ? 1 : 0;
        float incl = z;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const float Z = __shfl_sync(0xffffffffu, incl, 31);
        const float t = u * Z;
        const unsigned hit = __ballot_sync(0xffffffffu, (uint32_t)lane < G && incl > t);
        const unsigned nz = __ballot_sync(0xffffffffu, (uint32_t)lane < G && z > 0.f);
        int owner = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : -1);
        const float excl = __shfl_sync(0xffffffffu, incl - z, owner < 0 ? 0 : owner);
        if (lane == 0) {
            sc.bi[0] = (Z > 0.f && !any_fail) ? owner : -1;
            sc.bi[1] = hit ? 0 : 1;  // 1: take the last non-zero element of the owner
            sc.bi[3] = any_fail;
            sc.bf[0] = t - excl;
            sc.bf[1] = Z;
        }
    }
    __syncthreads();
    DrawResult res{sc.bi[0], -1, sc.bf[1], sc.bi[3]};
    const bool take_last = sc.bi[1] != 0;
    const float t_loc = sc.bf[0];
    __syncthreads();
    ++phase;
    if (res.owner < 0 || (uint32_t)res.owner != cluster_rank()) return res;
    // ---- owner CTA: warp 0 narrows the target to a tile, a lane and an element
    if (warp == 0) {
        int tile = -1, last_nz_tile = -1;
        float t_tile = 0.f;
        float cum = 0.f;
        for (int base = 0; base < ntiles && tile < 0; base += 32) {
            const float v = (base + lane < ntiles) ? tile_sum[base + lane] : 0.f;
            float incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const unsigned nzb = __ballot_sync(0xffffffffu, v > 0.f);
            if (nzb) last_nz_tile = base + 31 - __clz(nzb);
            const unsigned h = take_last ? 0u : __ballot_sync(0xffffffffu, cum + incl > t_loc);
            if (h) {
                const int f = __ffs(h) - 1;
                tile = base + f;
                t_tile = t_loc - (cum + __shfl_sync(0xffffffffu, incl - v, f));
            }
            cum += __shfl_sync(0xffffffffu, incl, 31);
        }
        bool last_mode = take_last;
        if (tile < 0) {
            tile = last_nz_tile;
            last_mode = true;
        }
        int token = -1;
        if (tile >= 0) {
            const int e0 = lo + tile * TILE + lane * VEC;
            float w[VEC];
            wf.eval8(e0, hi, w);
            const float ls = sum8(w);
            float incl = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const unsigned h = last_mode ? 0u : __ballot_sync(0xffffffffu, incl > t_tile);
            const unsigned nzl = __ballot_sync(0xffffffffu, ls > 0.f);
            int f;
            bool lane_last = last_mode;
            if (h) {
                f = __ffs(h) - 1;
            } else {
                f = nzl ? 31 - __clz(nzl) : 0;
                lane_last = true;
            }
            const float t_lane = t_tile - __shfl_sync(0xffffffffu, incl - ls, f);
            if (lane == f) {
                int pick = -1, last_nz = -1;
                float run = 0.f;
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (w[j] > 0.f) last_nz = j;
                    run += w[j];
                    if (!lane_last && pick < 0 && run > t_lane) pick = j;
                }
                if (pick < 0) pick = last_nz < 0 ? 0 : last_nz;
                token = e0 + pick;
            }
            token = __shfl_sync(0xffffffffu, token, f);
        }
        if (lane == 0) sc.bi[2] = token;
    }
    __syncthreads();
    res.token = sc.bi[2];
    __syncthreads();
    return res;
}

// Warp totals of TB per-lane values (TB = 1, 2 or 4), written to tile_sum[t0 + i] for the
// tiles below ntiles.  For TB > 1 the values are reduced transposed: each exchange step
// halves the values a lane keeps, so TB totals take TB - 1 + 5 - log2(TB) shuffles instead
// of 5 TB.
template <int TB>
__device__ __forceinline__ void warp_tile_sums(const float s[TB], int lane, int t0, int ntiles, float* tile_sum) {
    static_assert(TB == 1 || TB == 2 || TB == 4, "tiles in flight: 1, 2 or 4");
    float k;
    int i;
    if (TB == 1) {
        k = s[0];
        i = 0;
    } else if (TB == 2) {
        const bool b16 = (lane & 16) != 0;
        k = (b16 ? s[TB - 1] : s[0]) + __shfl_xor_sync(0xffffffffu, b16 ? s[0] : s[TB - 1], 16);
        i = b16 ? 1 : 0;
    } else {
        const bool b16 = (lane & 16) != 0, b8 = (lane & 8) != 0;
        // lanes without bit 4 of the lane index set keep tiles 0 and 1, the others 2 and 3
        float k0 = b16 ? s[2 % TB] : s[0], k1 = b16 ? s[3 % TB] : s[1 % TB];
        k0 += __shfl_xor_sync(0xffffffffu, b16 ? s[0] : s[2 % TB], 16);
        k1 += __shfl_xor_sync(0xffffffffu, b16 ? s[1 % TB] : s[3 % TB], 16);
        // then lanes without bit 3 keep the even tile of their pair, the others the odd one
        k = (b8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b8 ? k0 : k1, 8);
        i = (b16 ? 2 : 0) + (b8 ? 1 : 0);
    }
    // the lanes sharing a tile differ in the remaining low bits
#pragma unroll
    for (int o = (TB == 1 ? 16 : (TB == 2 ? 8 : 4)); o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
    const int width = 32 / TB;  // lanes per tile after the transposed steps
    if (lane % width == 0 && t0 + i < ntiles) tile_sum[t0 + i] = k;
}

// Tiles a warp evaluates before reducing them: weight functors that read global memory
// declare kTilesInFlight (several loads in flight per lane); shared-memory ones take 1.
template <class T, class = void>
struct TilesInFlight {
    static constexpr int value = 1;
};
template <class T>
struct TilesInFlight<T, decltype((void)T::kTilesInFlight)> {
    static constexpr int value = T::kTilesInFlight;
};

// Weight functors whose eval8_full(e0, w) evaluates eight elements that all lie below the
// end of the range (no bounds tests) use it for the draw's full tiles.
template <class T, class = void>
struct HasFullEval {
    static constexpr bool value = false;
};
template <class T>
struct HasFullEval<T, decltype((void)&T::eval8_full)> {
    static constexpr bool value = true;
};

template <class WF>
__device__ __forceinline__ void eval8_any(const WF& wf, int e0, int hi, bool full, float w[VEC]) {
    if constexpr (HasFullEval<WF>::value) {
        if (full) {
            wf.eval8_full(e0, w);
            return;
        }
    }
    wf.eval8(e0, hi, w);
}

// A weight functor with TB tiles in flight per warp, for kernels whose draw is bound by
// latency rather than by the exp2 pipe (one CTA per SM).
template <class WF, int TB>
struct InFlight : WF {
    static constexpr int kTilesInFlight = TB;
};

template <class WF, class SC>
__device__ DrawResult cluster_draw(const WF& wf, int lo, int hi, float u, float* tile_sum, SC& sc,
                                   int& phase, int fail_in = 0) {
    constexpr int TB = TilesInFlight<WF>::value;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);  // warps of this CTA
    const int ntiles = (hi - lo + TILE - 1) / TILE;
    const int nfull = (hi - lo) / TILE;  // tiles with no element at or beyond hi
    // each warp takes a contiguous run of tiles (runs differ by at most one tile), TB at a time
    const int w_lo = (warp * ntiles) / nw, w_hi = ((warp + 1) * ntiles) / nw;
    for (int t0 = w_lo; t0 < w_hi; t0 += TB) {
        float s[TB];  // each tile's weights are summed as soon as they are evaluated
#pragma unroll
        for (int i = 0; i < TB; ++i) {
            s[i] = 0.f;
            if (t0 + i < w_hi) {
                float w[VEC];
                eval8_any(wf, lo + (t0 + i) * TILE + lane * VEC, hi, t0 + i < nfull, w);
                s[i] = sum8(w);
            }
        }
        warp_tile_sums<TB>(s, lane, t0, w_hi, tile_sum);
    }
    __syncthreads();
    return cluster_draw_from_tiles(wf, lo, hi, u, tile_sum, sc, phase, fail_in);
}

}  // namespace sv
