// sv_internal.h -- argument blocks and launchers shared by the host entry points
// (sv_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace sv {

// Records a CUDA error for spec_verify_last_cuda_error (per calling thread), clears
// the sticky launch error and returns SV_ERR_CUDA; cudaSuccess gives SV_OK.
sv_status launch_status(cudaError_t e);

// out_count value of a batch row whose kernel gave up a bounded wait (a bulk copy or
// a cluster exchange that did not complete in time); 0 marks invalid data.
constexpr int32_t SV_COUNT_TIMEOUT = -1;

struct ChainArgs {
    const void* target;        // [B][K+1][V]
    const void* draft;         // [B][K][V] probs (fp32) or logits
    const int32_t* tokens;     // [B][K]
    const float* temperature;  // [B]; nullptr: every row greedy
    int B, K, V;
    uint64_t seed, offset;
    int32_t* out_tokens;       // [B][K+1]
    int32_t* out_count;        // [B]
    float* out_accept_prob;    // [B][K] or nullptr
    // Test hook of the staged walk (SPEC_VERIFY_TEST_STALL): batch row `stall_row` arms
    // its first copy barrier without issuing the copy, so that its bounded wait runs out
    // after `stall_ns`; -1 (the default) disables it.
    int stall_row = -1;
    uint32_t stall_ns = 0;
};

struct TreeArgs {
    const void* target;        // [B][N+1][V]
    const void* draft;         // [B][N+1][V]
    const int32_t* node_tokens;
    const int32_t* parent;
    const float* temperature;
    int B, N, V, max_depth;
    uint64_t seed, offset;
    int32_t* out_tokens;       // [B][D+1]
    int32_t* out_count;        // [B]
    int32_t* out_path;         // [B][D]
    int sibling_rule;          // SV_SIBLINGS_WITHOUT_REPLACEMENT or SV_SIBLINGS_IID
};

struct SampleArgs {
    const void* draft;         // [B][K][V] draft logits
    const float* temperature;  // [B]
    int B, K, V;
    uint64_t seed, offset;
    int32_t* out_draft_tokens; // [B][K]
};

// Positions (K + 1) the position-parallel chain kernel takes: its per-row counter word
// carries a reject bit and an invalid bit per position.
constexpr int SPEC_MAX_POS = 26;

// Per-tree arrays of the staged tree kernel in dynamic shared memory (N nodes): tokens,
// parents, children / depth counts, jump targets, accept uniforms (N each), draw
// uniforms (N + 1) and the rejection history (tried token, applied flag: N each;
// 1/Z and q scale: N + 1 each), rounded up to 128 bytes.
__host__ __device__ inline size_t tree_array_bytes(int N) {
    return ((size_t)(10 * N + 3) * 4 + 127) & ~(size_t)127;
}

// Largest chunk of a row a CTA of a G-CTA cluster owns (whole 8-element vectors).
__host__ __device__ inline int chunk_cap(int V, int G) {
    const int nvec = (V + 7) / 8;
    return ((nvec + G - 1) / G) * 8;
}

// Working area of the staged tree kernel: the current weights (fp32, one chunk) and
// the bitmask of tokens tried at the current node, 16-byte aligned.
__host__ __device__ inline size_t tree_work_bytes(int V, int G) {
    const size_t cap = (size_t)chunk_cap(V, G);
    return ((cap * 4 + 15) & ~(size_t)15) + ((((cap + 31) / 32) * 4 + 15) & ~(size_t)15);
}

// Shared-memory layout of the staged chain kernel (host-computed per launch).
struct StageLayout {
    int nslot;        // ring slots, one position's row chunks each (1..16)
    int slot_bytes;   // bytes per slot: target chunk + draft-logit chunk, 16-byte multiples
    int t_bytes;      // offset of the draft chunk inside a slot
    int probs_bytes;  // separate area for the rejected position's draft-probability chunk
    int prefetch_l2;  // prefetch the draft-probability chunks into L2 at kernel start
    int d_direct;     // draft-logit rows are read from global memory, not staged (slots hold the target only)
};

constexpr int STAGE_HEADER = 512;        // mbarriers (up to 2 * 16 + 1) at the start of dynamic shared memory
constexpr int MAX_DYN_SMEM = 227 * 1024; // opt-in dynamic shared memory per CTA on sm_103a

size_t staged_smem_bytes(const StageLayout& L, int V, int G);
cudaError_t launch_chain_staged(const ChainArgs& a, const StageLayout& L, int tdt, int ddt, int dk, int cluster,
                                cudaStream_t stream);

cudaError_t launch_tree_staged(const TreeArgs& a, const StageLayout& L, int tdt, int ddt, int dk, int cluster,
                               cudaStream_t stream);

// Ring-streamed walk for large batches (sv_chain_ring.cu): every row resident, each
// CTA's chunk streamed through `nstage` stages of 2048 elements (target piece, then the
// draft piece at byte t_bytes).
struct RingLayout {
    int nstage;       // stages in the ring (1..8)
    int stage_bytes;  // bytes per stage, 16-byte multiple
    int t_bytes;      // offset of the draft piece inside a stage
};
size_t ring_smem_bytes(const RingLayout& L, int V, int G);
cudaError_t launch_chain_ring(const ChainArgs& a, const RingLayout& L, int tdt, int ddt, int dk, int cluster,
                              cudaStream_t stream);

// All-positions-at-once chain kernel (small batches, K + 1 <= 16).
cudaError_t launch_chain_eager(const ChainArgs& a, int tdt, int ddt, int dk, int cluster, cudaStream_t stream);

// Position-parallel chain kernel (small batches): workspace bytes and launch.
size_t spec_workspace_bytes(int B, int K, int V, int G);
size_t spec_smem_bytes(int V, int G, int tsz, int dsz, int* t_bytes, int* d_bytes);
cudaError_t launch_chain_spec(const ChainArgs& a, void* ws, int tdt, int ddt, int dk, int cluster, cudaStream_t stream);

// spec_verify_chain with the workspace supplied by the library itself (used by the
// entry point that allocates nothing).
sv_status chain_with_scratch(const void* target_logits, int tdt, const void* draft, int ddt, int dk,
                             const int32_t* draft_tokens, const float* temperature, int B, int K, int V,
                             uint64_t seed, uint64_t offset, int32_t* out_tokens, int32_t* out_count,
                             float* out_accept_prob, void* scratch, size_t scratch_bytes, void* stream);

// Cluster size (CTAs per batch row) for a launch over B batch rows.
int choose_cluster(int B, int V, int num_sms);

cudaError_t launch_chain(const ChainArgs& a, int tdt, int ddt, int dk, int cluster, cudaStream_t stream);
cudaError_t launch_tree(const TreeArgs& a, int tdt, int ddt, int dk, int cluster, cudaStream_t stream);

// Dynamic shared memory (tile sums of the draw) for a row split `cluster` ways.
size_t draw_smem_bytes(int V, int cluster);


// Launch facts of one kernel, kept per device ordinal and filled under a mutex, so
// that several host threads and several devices may launch it: the kernel's function
// attributes are set on each device on first use there (cluster sizes above 8, the
// opt-in dynamic shared memory), and occupancy answers are cached per launch shape.
class KernelLaunchCache {
public:
    // Sets the kernel up on the current device (once) and returns in *max_dyn the
    // dynamic shared memory it may request there (opt-in limit minus its static part).
    cudaError_t setup(const void* kern, int* max_dyn);
    // Largest cluster the current device co-schedules for a launch with cfg's block
    // size and dynamic shared memory (cudaOccupancyMaxPotentialClusterSize); 0 when
    // that shared memory is beyond the kernel's limit.
    cudaError_t max_cluster(const void* kern, const cudaLaunchConfig_t& cfg, int* out);
    // Clusters of G CTAs resident at once for that launch shape (cudaOccupancyMaxActiveClusters).
    cudaError_t active_clusters(const void* kern, const cudaLaunchConfig_t& cfg, int G, int* out);
    // The cluster size to launch a kernel whose dynamic shared memory depends on it
    // (smem_for(G)): the requested size when the device co-schedules it with that memory,
    // else the nearest smaller size that it does, else the nearest larger one (a larger
    // cluster gives each CTA a smaller chunk).  *G is 0 when no size up to 16 fits.
    template <class SmemFor>
    cudaError_t pick_cluster(const void* kern, cudaLaunchConfig_t cfg, int want, SmemFor smem_for, int* G) {
        *G = 0;
        int cand[10], nc = 0;
        for (int g = want; g >= 1; g >>= 1) cand[nc++] = g;
        for (int g = want * 2; g <= 16; g <<= 1) cand[nc++] = g;
        for (int i = 0; i < nc; ++i) {
            cfg.dynamicSmemBytes = smem_for(cand[i]);
            int maxc = 0;
            const cudaError_t e = max_cluster(kern, cfg, &maxc);
            if (e != cudaSuccess) return e;
            if (maxc >= cand[i]) {
                *G = cand[i];
                return cudaSuccess;
            }
        }
        return cudaSuccess;
    }

private:
    static constexpr int kDevices = 64;
    static constexpr int kEntries = 8;
    struct Entry {
        size_t smem;
        unsigned threads;
        int G;  // 0: max_cluster entry
        int value;
    };
    struct Device {
        bool ready = false;
        int max_dyn = 0;
        int used = 0;
        Entry e[kEntries];
    };
    cudaError_t device(const void* kern, Device** out);
    std::mutex mu_;
    Device dev_[kDevices];
};

// Draft tokens x_k ~ softmax(draft_k / T) (argmax for greedy rows) for every (b, k).
cudaError_t launch_draft_sample(const SampleArgs& a, int ddt, int num_sms, cudaStream_t stream);

}  // namespace sv
