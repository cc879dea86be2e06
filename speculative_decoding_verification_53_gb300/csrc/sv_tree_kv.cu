// sv_tree_kv.cu -- the steps on either side of a tree verify (include/spec_tree_kv.h):
// the ancestor-or-self attention mask of a draft tree, and the compaction of the
// accepted branch's KV-cache rows into a contiguous prefix.
//
// Tree mask ("Speculative Decoding and EAGLE", section "트리 어텐션 검증": every
// token attends to its ancestors in the tree, and to itself as in any causal
// mask).  One CTA per batch row.  Depths first, by pointer jumping on (count,
// jump target) pairs: ceil(log2(depth)) + 1 rounds, each reading everything it
// needs, synchronising, then writing.  Then the nodes are bucketed by depth and
// the rows filled level by level, row(i) = row(parent(i)) | bit(i): every word is
// computed once, kept in shared memory for the children and stored straight to
// HBM in 16-byte chunks (a warp writes whole rows).  Shared rows are triangular,
// so a tree of 1024 nodes needs 90 KB and two CTAs share an SM.  Trees deeper
// than 64 levels fill the rows by pointer jumping instead (log rounds rather than
// one barrier per level), then copy them out.  Trees of at most 64 nodes take a
// warp each and do the pointer jumping on 64-bit rows in registers.
//
// KV compaction ("[논문 리뷰] Fast Inference from Transformers via Speculative
// Decoding", section 4: rejected tokens' cache entries must be rolled back).  A
// path's node indices increase along it, so path[d] >= d and no source row is a
// destination of an earlier copy: the in-order copies equal a gather from the
// cache as it was.  So every thread owns one aligned piece (16, 4 or 1 bytes) of
// one (buffer, plane) row slot and moves that piece for every accepted depth,
// loading up to eight sources before storing them.  The work is pure HBM traffic:
// 2 x row_bytes per moved row and plane.
#include <cstdint>

#include "spec_tree_kv.h"
#include "sv_common.cuh"
#include "sv_internal.h"

namespace {

using sv::pdl_trigger;
using sv::pdl_wait;

// A launch with programmatic stream serialization (the kernels call pdl_wait first).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kMaskMaxN = 1024;
constexpr int kKvMaxBuffers = 256;
constexpr int kKvMaxDepth = 64;
constexpr int kKvThreads = 256;
constexpr int kKvBatch = 8;  // sources loaded before their stores

// ------------------------------------------------------------------ tree mask

constexpr int kMaskLevelMaxDepth = 64;  // deeper trees take the pointer-jumping pass

// Shared-memory rows are triangular: row i holds only words 0 .. i/32 (its
// ancestors precede it), padded to a multiple of four words so that every row and
// 16-byte chunk is aligned.  Row i starts at tri_off(i); rows of the same 32-node
// block c have tri_len(c) words.
__device__ __forceinline__ int tri_len(int c) { return (c + 4) & ~3; }
__device__ __forceinline__ int tri_off(int i) {
    const int c = i >> 5, q = c >> 2, m = c & 3;
    return 256 * q * (q + 1) + 128 * m * (q + 1) + (i & 31) * tri_len(c);
}

__device__ __forceinline__ uint4 ld_chunk(const uint32_t* s, int off) {
    return *reinterpret_cast<const uint4*>(s + off);
}
__device__ __forceinline__ void st_chunk(uint32_t* s, int off, uint4 v) { *reinterpret_cast<uint4*>(s + off) = v; }

// Stores chunk q (words 4q .. 4q+3) of an output row of W words.
__device__ __forceinline__ void store_out_chunk(uint32_t* row, int W, int q, uint4 v) {
    const int w0 = 4 * q;
    if (w0 + 4 <= W && (W & 3) == 0) {
        *reinterpret_cast<uint4*>(row + w0) = v;
    } else {
        if (w0 + 0 < W) row[w0 + 0] = v.x;
        if (w0 + 1 < W) row[w0 + 1] = v.y;
        if (w0 + 2 < W) row[w0 + 2] = v.z;
        if (w0 + 3 < W) row[w0 + 3] = v.w;
    }
}

__device__ __forceinline__ void set_bit(uint4& v, int word_in_chunk, uint32_t bit) {
    if (word_in_chunk == 0) v.x |= bit;
    else if (word_in_chunk == 1) v.y |= bit;
    else if (word_in_chunk == 2) v.z |= bit;
    else v.w |= bit;
}

// CW: 16-byte chunks an output row needs, rounded up to a power of two (1..8).  A
// warp handles 32 / CW nodes at a time, lane (lane % CW) owning chunk q of a row.
template <int CW>
__global__ void __launch_bounds__(1024, 2) tree_mask_kernel(const int32_t* __restrict__ parent, int N, int W,
                                                            uint32_t* __restrict__ out_mask,
                                                            int32_t* __restrict__ out_depth,
                                                            int32_t* __restrict__ out_valid) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    extern __shared__ __align__(16) uint32_t s_rows[];
    int* s_par = reinterpret_cast<int*>(s_rows + tri_off(N));
    int* s_dep = s_par + N;    // nodes from i up to its current jump target (finally: the depth)
    int* s_jump = s_dep + N;
    int* s_order = s_jump + N;  // node ids sorted by depth
    __shared__ int s_off[kMaskLevelMaxDepth + 2], s_cur[kMaskLevelMaxDepth + 2];
    __shared__ int s_maxd;
    const int b = blockIdx.x, i = threadIdx.x, lane = i & 31, warp = i >> 5, nwarps = blockDim.x >> 5;
    const bool is_node = i < N;
    const size_t words = (size_t)N * W;
    uint32_t* mask_b = out_mask + (size_t)b * words;
    constexpr int G = 32 / CW;
    const int sub = lane / CW, q = lane % CW;

    const int p = is_node ? __ldg(parent + (size_t)b * N + i) : -1;
    if (__syncthreads_or(is_node && (p < -1 || p >= i))) {
        for (size_t f = i; f < words; f += blockDim.x) mask_b[f] = 0u;
        if (is_node && out_depth) out_depth[(size_t)b * N + i] = 0;
        if (i == 0 && out_valid) out_valid[b] = 0;
        return;
    }
    if (i == 0) s_maxd = 0;
    for (int c = i; c < kMaskLevelMaxDepth + 2; c += blockDim.x) s_off[c] = 0;
    if (is_node) {
        s_par[i] = p;
        s_dep[i] = 1;
        s_jump[i] = p;
    }
    // Depths by pointer jumping on (count, target) pairs: read, barrier, write.
    int a = p, d = 1;
    while (__syncthreads_or(a >= 0)) {
        int da = 0, na = -1;
        if (a >= 0) {
            da = s_dep[a];
            na = s_jump[a];
        }
        __syncthreads();
        if (a >= 0) {
            d += da;
            a = na;
            s_dep[i] = d;
            s_jump[i] = a;
        }
    }
    if (is_node && out_depth) out_depth[(size_t)b * N + i] = d;
    const int key = is_node ? d : -1;  // every lane of the block takes part below
    const int warp_max = __reduce_max_sync(0xffffffffu, key);
    if (lane == 0) atomicMax(&s_maxd, warp_max);
    __syncthreads();
    const int maxd = s_maxd;
    if (i == 0 && out_valid) out_valid[b] = 1;

    if (maxd <= kMaskLevelMaxDepth) {
        // Level order: bucket the nodes by depth (a warp's equal-depth nodes keep
        // their index order), then row(i) = row(parent(i)) | bit(i), level by level.
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (is_node && rank == 0) atomicAdd(&s_off[d + 1], __popc(peers));
        __syncthreads();
        if (warp == 0) {  // inclusive scan of the level counts (at most 66 bins)
            int carry = 0;
            for (int c0 = 0; c0 <= maxd + 1; c0 += 32) {
                const int c = c0 + lane;
                int v = c <= maxd + 1 ? s_off[c] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                v += carry;
                if (c <= maxd + 1) {
                    s_off[c] = v;
                    s_cur[c] = v;
                }
                carry = __shfl_sync(0xffffffffu, v, 31);
            }
        }
        __syncthreads();
        int pos = 0;
        if (is_node && rank == 0) pos = atomicAdd(&s_cur[d], __popc(peers));
        pos = __shfl_sync(0xffffffffu, pos, __ffs(peers) - 1) + rank;
        if (is_node) s_order[pos] = i;
        __syncthreads();
        for (int L = 1; L <= maxd; ++L) {
            const int lo = s_off[L], hi = s_off[L + 1];
            for (int k = lo + warp * G + sub; k < hi; k += nwarps * G) {
                const int node = s_order[k];
                const int par = s_par[node];
                const int top = node >> 5;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (q <= (top >> 2)) {  // chunk q is part of the node's shared row
                    if (par >= 0 && q <= ((par >> 5) >> 2)) v = ld_chunk(s_rows, tri_off(par) + 4 * q);
                    if ((top >> 2) == q) set_bit(v, top & 3, 1u << (node & 31));
                    st_chunk(s_rows, tri_off(node) + 4 * q, v);
                }
                if (4 * q < W) store_out_chunk(mask_b + (size_t)node * W, W, q, v);
            }
            __syncthreads();
        }
        return;
    }

    // Deep trees: pointer jumping on the rows.  Row i holds the nodes from i up to
    // (not including) its jump target; a round ORs in the target's row and jumps on.
    // Row a has nothing above word a >> 5, i.e. above chunk (a >> 5) >> 2.
    if (is_node) {
        const int top = i >> 5;
        for (int c = 0; c <= (top >> 2); ++c) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if ((top >> 2) == c) set_bit(v, top & 3, 1u << (i & 31));
            st_chunk(s_rows, tri_off(i) + 4 * c, v);
        }
        s_jump[i] = p;
    }
    a = p;
    while (__syncthreads_or(a >= 0)) {
        int next = -1, ctop = -1;
        if (a >= 0) {
            ctop = (a >> 5) >> 2;
            next = s_jump[a];
        }
        // Four passes of at most two chunks each keep the per-thread copy small.
        for (int h = 0; h < 4; ++h) {
            uint4 t[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int cc = 2 * h + c;
                t[c] = (a >= 0 && cc <= ctop) ? ld_chunk(s_rows, tri_off(a) + 4 * cc) : make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
            if (a >= 0) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int cc = 2 * h + c;
                    if (cc <= ctop) {
                        uint4 v = ld_chunk(s_rows, tri_off(i) + 4 * cc);
                        v.x |= t[c].x;
                        v.y |= t[c].y;
                        v.z |= t[c].z;
                        v.w |= t[c].w;
                        st_chunk(s_rows, tri_off(i) + 4 * cc, v);
                    }
                }
            }
            __syncthreads();
        }
        if (a >= 0) {
            a = next;
            s_jump[i] = a;
        }
    }
    for (int k = warp * G + sub; k < N; k += nwarps * G) {
        const int top = k >> 5;
        const uint4 v = (q <= (top >> 2)) ? ld_chunk(s_rows, tri_off(k) + 4 * q) : make_uint4(0u, 0u, 0u, 0u);
        if (4 * q < W) store_out_chunk(mask_b + (size_t)k * W, W, q, v);
    }
}

// Trees of at most 64 nodes: one warp per tree, no shared memory and no barrier.
// Lane l holds nodes l and l + 32, each with a 64-bit row (the nodes from it up
// to its jump target), the node count of that stretch and the target; a round
// fetches the targets' values with shuffles, all lanes reading the values of the
// previous round, so it is the same pointer jumping as above in registers.
constexpr int kSmallMaskTreesPerCta = 8;

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
    return ((uint64_t)hi << 32) | lo;
}

__global__ void __launch_bounds__(32 * kSmallMaskTreesPerCta) tree_mask_small_kernel(
    const int32_t* __restrict__ parent, int B, int N, int W, uint32_t* __restrict__ out_mask,
    int32_t* __restrict__ out_depth, int32_t* __restrict__ out_valid) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kSmallMaskTreesPerCta + (threadIdx.x >> 5);
    if (b >= B) return;  // whole warps leave together
    const int i0 = lane, i1 = lane + 32;
    const bool n0 = i0 < N, n1 = i1 < N;
    const int32_t* par_b = parent + (size_t)b * N;
    const int p0 = n0 ? __ldg(par_b + i0) : -1;
    const int p1 = n1 ? __ldg(par_b + i1) : -1;
    const bool bad = (n0 && (p0 < -1 || p0 >= i0)) || (n1 && (p1 < -1 || p1 >= i1));
    uint32_t* mask_b = out_mask + (size_t)b * N * W;
    if (__any_sync(0xffffffffu, bad)) {
        for (int f = lane; f < N * W; f += 32) mask_b[f] = 0u;
        if (out_depth) {
            if (n0) out_depth[(size_t)b * N + i0] = 0;
            if (n1) out_depth[(size_t)b * N + i1] = 0;
        }
        if (lane == 0 && out_valid) out_valid[b] = 0;
        return;
    }
    uint64_t m0 = n0 ? 1ull << i0 : 0ull, m1 = n1 ? 1ull << i1 : 0ull;
    int a0 = p0, a1 = p1, d0 = 1, d1 = 1;
    while (__any_sync(0xffffffffu, a0 >= 0 || a1 >= 0)) {
        // the values of node x live in lane x & 31, slot x >> 5
        const int s0 = a0 & 31, s1 = a1 & 31;
        const uint64_t ma0_lo = shfl_u64(m0, s0), ma0_hi = shfl_u64(m1, s0);
        const uint64_t ma1_lo = shfl_u64(m0, s1), ma1_hi = shfl_u64(m1, s1);
        const int da0_lo = __shfl_sync(0xffffffffu, d0, s0), da0_hi = __shfl_sync(0xffffffffu, d1, s0);
        const int da1_lo = __shfl_sync(0xffffffffu, d0, s1), da1_hi = __shfl_sync(0xffffffffu, d1, s1);
        const int aa0_lo = __shfl_sync(0xffffffffu, a0, s0), aa0_hi = __shfl_sync(0xffffffffu, a1, s0);
        const int aa1_lo = __shfl_sync(0xffffffffu, a0, s1), aa1_hi = __shfl_sync(0xffffffffu, a1, s1);
        if (a0 >= 0) {
            const bool hi = a0 >= 32;
            m0 |= hi ? ma0_hi : ma0_lo;
            d0 += hi ? da0_hi : da0_lo;
            a0 = hi ? aa0_hi : aa0_lo;
        }
        if (a1 >= 0) {
            const bool hi = a1 >= 32;
            m1 |= hi ? ma1_hi : ma1_lo;
            d1 += hi ? da1_hi : da1_lo;
            a1 = hi ? aa1_hi : aa1_lo;
        }
    }
    if (W == 1) {
        if (n0) mask_b[i0] = (uint32_t)m0;
    } else {
        if (n0) *reinterpret_cast<uint2*>(mask_b + 2 * i0) = make_uint2((uint32_t)m0, (uint32_t)(m0 >> 32));
        if (n1) *reinterpret_cast<uint2*>(mask_b + 2 * i1) = make_uint2((uint32_t)m1, (uint32_t)(m1 >> 32));
    }
    if (out_depth) {
        if (n0) out_depth[(size_t)b * N + i0] = d0;
        if (n1) out_depth[(size_t)b * N + i1] = d1;
    }
    if (lane == 0 && out_valid) out_valid[b] = 1;
}

size_t mask_smem_bytes(int N) {
    const int c = N >> 5, qq = c >> 2, m = c & 3;
    const size_t tri = 256 * (size_t)qq * (qq + 1) + 128 * (size_t)m * (qq + 1) + (size_t)(N & 31) * ((c + 4) & ~3);
    return (tri + 4 * (size_t)N) * sizeof(uint32_t);
}

template <int CW>
cudaError_t launch_mask(const int32_t* parent, int B, int N, int W, uint32_t* mask, int32_t* depth, int32_t* valid,
                        cudaStream_t stream) {
    const int threads = ((N + 31) / 32) * 32;
    const size_t smem = mask_smem_bytes(N);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(tree_mask_kernel<CW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(tree_mask_kernel<CW>, dim3(B), dim3(threads), smem, stream, parent, N, W, mask, depth, valid);
}

// ------------------------------------------------------------- KV compaction

struct KvArgs {
    unsigned char* buf[kKvMaxBuffers];
    int64_t batch_stride, plane_stride, row_stride;
    int num_buffers, num_planes, pieces;  // pieces: row_bytes / piece width
    int num_rows, D;
    const int32_t* path;
    const int32_t* count;
    const int32_t* base;
};

template <int PW> struct Piece;
template <> struct Piece<16> { using T = uint4; };
template <> struct Piece<4> { using T = uint32_t; };
template <> struct Piece<1> { using T = uint8_t; };

// grid: x covers num_buffers * num_planes * pieces, y is the batch row.
template <int PW>
__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(const __grid_constant__ KvArgs a) {
    pdl_trigger();
    pdl_wait();  // nothing the previous kernel on the stream writes is read before this
    using T = typename Piece<PW>::T;
    __shared__ int s_dst[kKvMaxDepth], s_src[kKvMaxDepth];
    __shared__ int s_moves, s_base;
    const int b = blockIdx.y;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int cnt = __ldg(a.count + b);
        const int L = cnt - 1;
        const int base = a.base ? __ldg(a.base + b) : 0;
        bool ok = cnt >= 1 && L <= a.D && base >= 0;
        int moves = 0;
        for (int d0 = 0; d0 < a.D; d0 += 32) {
            const int d = d0 + lane;
            int s = d;
            bool lane_ok = true;
            if (ok && d < L) {
                s = __ldg(a.path + (size_t)b * a.D + d);
                lane_ok = s >= d && (int64_t)base + s < a.num_rows;
            }
            ok = ok && __all_sync(0xffffffffu, lane_ok);
            const bool move = ok && d < L && s != d;  // a row already in place is not copied
            const unsigned m = __ballot_sync(0xffffffffu, move);
            if (move) {
                const int slot = moves + __popc(m & ((1u << lane) - 1u));
                s_dst[slot] = d;
                s_src[slot] = s;
            }
            moves += __popc(m);
        }
        if (lane == 0) {
            s_moves = ok ? moves : 0;
            s_base = base;
        }
    }
    __syncthreads();
    const int moves = s_moves;
    const unsigned f = blockIdx.x * kKvThreads + threadIdx.x;
    const unsigned total = (unsigned)a.num_buffers * a.num_planes * a.pieces;
    if (moves == 0 || f >= total) return;
    const unsigned piece = f % a.pieces, rest = f / a.pieces;
    const unsigned h = rest % a.num_planes, k = rest / a.num_planes;
    unsigned char* p0 = a.buf[k] + (int64_t)b * a.batch_stride + (int64_t)h * a.plane_stride +
                        (int64_t)s_base * a.row_stride + (int64_t)piece * PW;
    for (int m0 = 0; m0 < moves; m0 += kKvBatch) {
        T v[kKvBatch];
#pragma unroll
        for (int j = 0; j < kKvBatch; ++j)
            if (m0 + j < moves) v[j] = *reinterpret_cast<const T*>(p0 + (int64_t)s_src[m0 + j] * a.row_stride);
#pragma unroll
        for (int j = 0; j < kKvBatch; ++j)
            if (m0 + j < moves) *reinterpret_cast<T*>(p0 + (int64_t)s_dst[m0 + j] * a.row_stride) = v[j];
    }
}

}  // namespace

extern "C" {

sv_status spec_tree_mask(const int32_t* parent, int B, int N, uint32_t* out_mask, int32_t* out_depth,
                         int32_t* out_valid, void* stream) {
    if (B < 0 || B > 65535 || N < 1 || N > kMaskMaxN) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!parent || !out_mask) return SV_ERR_INVALID_ARG;
    const int W = (N + 31) / 32;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    const int chunks = (W + 3) / 4;
    if (N <= 64) {
        const int grid = (B + kSmallMaskTreesPerCta - 1) / kSmallMaskTreesPerCta;
        e = launch_pdl(tree_mask_small_kernel, dim3(grid), dim3(32 * kSmallMaskTreesPerCta), 0, s, parent, B, N, W,
                       out_mask, out_depth, out_valid);
    } else if (chunks <= 1) e = launch_mask<1>(parent, B, N, W, out_mask, out_depth, out_valid, s);
    else if (chunks <= 2) e = launch_mask<2>(parent, B, N, W, out_mask, out_depth, out_valid, s);
    else if (chunks <= 4) e = launch_mask<4>(parent, B, N, W, out_mask, out_depth, out_valid, s);
    else e = launch_mask<8>(parent, B, N, W, out_mask, out_depth, out_valid, s);
    return sv::launch_status(e);
}

sv_status spec_kv_compact(void* const* kv_buffers, int num_buffers, int64_t batch_stride, int64_t plane_stride,
                          int num_planes, int64_t row_stride, int64_t row_bytes, int num_rows, const int32_t* path,
                          const int32_t* count, const int32_t* base, int B, int max_depth, void* stream) {
    if (B < 0 || B > 65535 || num_buffers < 1 || num_buffers > kKvMaxBuffers || num_planes < 1 ||
        max_depth < 1 || max_depth > kKvMaxDepth || num_rows < 1 || row_bytes < 1 || row_stride < row_bytes ||
        batch_stride < 0 || plane_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!kv_buffers || !path || !count) return SV_ERR_INVALID_ARG;
    KvArgs a{};
    uint64_t align = (uint64_t)batch_stride | (uint64_t)plane_stride | (uint64_t)row_stride | (uint64_t)row_bytes;
    for (int k = 0; k < num_buffers; ++k) {
        if (!kv_buffers[k]) return SV_ERR_INVALID_ARG;
        a.buf[k] = static_cast<unsigned char*>(kv_buffers[k]);
        align |= (uint64_t)(uintptr_t)kv_buffers[k];
    }
    const int pw = (align % 16 == 0) ? 16 : (align % 4 == 0) ? 4 : 1;
    const int64_t pieces = row_bytes / pw;
    const int64_t total = (int64_t)num_buffers * num_planes * pieces;
    if (total > (int64_t)INT32_MAX - kKvThreads) return SV_ERR_INVALID_ARG;
    a.batch_stride = batch_stride;
    a.plane_stride = plane_stride;
    a.row_stride = row_stride;
    a.num_buffers = num_buffers;
    a.num_planes = num_planes;
    a.pieces = (int)pieces;
    a.num_rows = num_rows;
    a.D = max_depth;
    a.path = path;
    a.count = count;
    a.base = base;
    const dim3 grid((unsigned)((total + kKvThreads - 1) / kKvThreads), (unsigned)B);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (pw == 16) e = launch_pdl(kv_compact_kernel<16>, grid, dim3(kKvThreads), 0, s, a);
    else if (pw == 4) e = launch_pdl(kv_compact_kernel<4>, grid, dim3(kKvThreads), 0, s, a);
    else e = launch_pdl(kv_compact_kernel<1>, grid, dim3(kKvThreads), 0, s, a);
    return sv::launch_status(e);
}

}  // extern "C"
