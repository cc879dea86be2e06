/*
 * spec_tree_kv.h -- the two steps around a tree verify: the tree-attention mask the
 * target's verify pass needs before it runs, and the KV-cache compaction that
 * keeps only the accepted branch after it.  Same library, status codes and
 * conventions as spec_verify.h (caller-owned device arrays, asynchronous on
 * `stream`, argument errors returned before any launch, SV_ERR_CUDA for launch
 * failures).
 *
 * Defining passages (page title, section):
 *  - "Speculative Decoding and EAGLE", section "트리 어텐션 검증 (Tree Attention
 *    Verification)": the target checks the whole draft tree in one forward pass
 *    under a causal mask that encodes the tree, in which each token attends only
 *    to its ancestors; the same page's project description lists a builder of
 *    that mask.
 *  - "Progressive Tree Drafting" summary, sections "트리 구조 드래프팅" and "검증":
 *    the attention mask and the position encoding are rebuilt so that one forward
 *    pass follows every branch of the tree.
 *  - "[논문 리뷰] Fast Inference from Transformers via Speculative Decoding",
 *    section 4 "한계점": the KV-cache entries of rejected tokens must be rolled
 *    back, which the review names as a source of implementation complexity.
 */
#ifndef SPEC_TREE_KV_H
#define SPEC_TREE_KV_H

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Tree-attention mask: for every node of every batch row, the set of tree nodes it
 * may attend to, namely itself and its ancestors (the root and the context before
 * it are visible to every node and are not part of the mask).
 *   parent      device int32 [B][N], parent[i] in {-1} u [0, i) (-1: child of the
 *               root) -- the layout spec_verify_tree takes.  1 <= N <= 1024.
 *   out_mask    device uint32 [B][N][W], W = ceil(N / 32): bit (j % 32) of word
 *               j / 32 of row i is set iff node j is node i or an ancestor of it.
 *               Bits at positions >= N are clear.
 *   out_depth   device int32 [B][N] or NULL: the number of nodes on the path from
 *               the root's child down to node i (1 for a child of the root), that
 *               is the number of set bits of row i; the node's position id is the
 *               root's position plus its depth.
 *   out_valid   device int32 [B] or NULL: 1, or 0 for a batch row whose parent
 *               array is malformed; that row's mask and depths are all zero.
 * Errors: SV_ERR_INVALID_ARG for B < 0, B > 65535, N outside [1, 1024] or a NULL
 * parent / out_mask (B = 0 returns SV_OK and launches nothing).
 */
SV_API sv_status spec_tree_mask(const int32_t *parent, int B, int N,
                                uint32_t *out_mask, int32_t *out_depth, int32_t *out_valid,
                                void *stream);

/*
 * Accepted-path KV compaction.  In a tree verify pass, node i of batch row b wrote
 * its key/value vectors at cache row base[b] + i.  The accepted nodes path[b][0..L-1]
 * (L = count[b] - 1: the last emitted token is not in the cache yet) are moved to
 * rows base[b] + 0 .. base[b] + L - 1, in path order, so the next round continues
 * from a contiguous prefix.  The move has the meaning of the in-order copies
 * "for d = 0..L-1: row base+d <- row base+path[d]"; because path[d] >= d (a path's
 * node indices increase along it), this equals gathering every source from the
 * cache as it was before the call.  Rows that are not destinations keep their
 * bytes.  path and count are spec_verify_tree's out_path and out_count.
 *
 *   kv_buffers   HOST array of num_buffers device pointers (one per cache tensor,
 *                e.g. each layer's K and V); read during the call and captured into
 *                the launch, so the host array may be reused afterwards.
 *                1 <= num_buffers <= 256.
 *   batch_stride, plane_stride, row_stride   byte strides: row r of batch row b and
 *                plane h (a KV head) of buffer k starts at
 *                kv_buffers[k] + b*batch_stride + h*plane_stride + r*row_stride.
 *   num_planes   >= 1;  row_bytes: bytes per (plane, row), 1 <= row_bytes <= row_stride.
 *   num_rows     cache rows per plane (a source or destination at or beyond it makes
 *                the batch row invalid).
 *   path         device int32 [B][max_depth], -1 padded; count device int32 [B];
 *   base         device int32 [B] or NULL (every base 0).  1 <= max_depth <= 64.
 * A batch row with count 0 (an invalid verify row), count > max_depth + 1, an entry
 * path[d] < d, a negative base or a row at or beyond num_rows is left untouched.
 * The copies use 16-byte accesses when every pointer, stride and row_bytes is a
 * multiple of 16, else 4- or 1-byte ones.  Buffers, planes and batch rows must
 * not overlap one another.
 * Errors: SV_ERR_INVALID_ARG for a bad size, a NULL pointer among kv_buffers, path
 * or count, or row_bytes > row_stride (B = 0 returns SV_OK).
 */
SV_API sv_status spec_kv_compact(void *const *kv_buffers, int num_buffers,
                                 int64_t batch_stride, int64_t plane_stride, int num_planes,
                                 int64_t row_stride, int64_t row_bytes, int num_rows,
                                 const int32_t *path, const int32_t *count, const int32_t *base,
                                 int B, int max_depth, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_KV_H */
