/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding verify library.
 *
 * The library implements the target-side verify/accept step of speculative
 * decoding: given the target model's logits at the K+1 drafted positions, the
 * draft distribution and the K drafted tokens, it decides which drafted tokens
 * are kept and emits one more token (a replacement or a bonus token).
 *
 * Defining passages (page title, section):
 *  - "[논문 리뷰] Fast Inference from Transformers via Speculative Decoding"
 *    (review of Leviathan et al., ICML 2023), section 2 "제안 방법": Step 3
 *    "Accept/Reject" (left to right, acceptance probability min(1, p(x)/q(x)),
 *    replacement from max(0, p-q)/sum max(0, p-q) at the first rejection, later
 *    drafts discarded, 1..K+1 tokens per round).
 *  - "Speculative Decoding and EAGLE", sections "개념" (bonus token when all K
 *    pass) and "정확성 규칙 (The Exactness Rule)" (r < p/q; residual
 *    (p-q)+/||(p-q)+||_1; the greedy case accepts iff argmax(p) == x_t, else
 *    emits argmax(p) and stops); section "트리 어텐션 검증" (the longest
 *    accepted branch of a draft tree).
 *  - "Progressive Tree Drafting" summary, section "검증 (Verification)":
 *    greedy tree acceptance (an edge is accepted when the verified token equals
 *    a child) and sampling acceptance without replacement from normalised
 *    probabilities.
 *
 * Conventions shared by every entry point
 *  - Pointers named as device arrays are caller-owned device memory; the library
 *    never allocates, frees or retains them.  Arrays are dense and row-major in
 *    the order their shapes are written.  Logits may be fp32 or bf16 (SV_F32 /
 *    SV_BF16); draft probabilities are fp32.
 *  - p = softmax(logits / T) per row; T <= 0 (or NaN) selects the greedy rule for
 *    that batch row.  A draft given as logits uses the same T; a draft given as
 *    probabilities is used as given (it must be a distribution).
 *  - Randomness: Philox4x64-10 with counter {slot, b, offset, 0} and key
 *    {seed, 0}, b the batch row index within the call.  Word 0 of slot k is the
 *    accept uniform of chain position k (tree: of node k); word 1 of slot k is the
 *    draw uniform at chain position k (tree: at distribution row k).  A uniform
 *    is (w >> 40) * 2^-24.  The caller advances `offset` (or `seed`) per round.
 *  - Acceptance is r < p(x)/q(x); q(x) == 0 accepts iff p(x) > 0.  Replacement
 *    and bonus draws are inverse-CDF draws: the smallest index i whose prefix
 *    sum C_i exceeds u * Z, Z the total weight.  A residual with zero mass falls
 *    back to p.  argmax ties resolve to the lowest index.
 *  - Arithmetic is fp32 on the device.  Results match an fp64 evaluation of the
 *    same rule except where a decision lies within fp32 rounding of its boundary.
 *  - Execution is asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream).  Argument errors are detected on the host and
 *    returned before anything is launched.  Launch failures return SV_ERR_CUDA.
 *  - Per-row data errors do not fail the call: a batch row whose read logits
 *    contain NaN or +inf or are all -inf, whose tokens lie outside [0, V), whose
 *    draft probability at a drafted token is negative or not finite, or whose
 *    parent array is malformed, gets out_count[b] = 0 and all output slots -1.
 *    A valid row always has out_count[b] >= 1.
 *  - Every device-side wait (for a bulk copy, or for the partial results the CTAs of
 *    a thread-block cluster exchange) is bounded to a quarter of a second.  A wait
 *    that gives up does not fail the call either: the walking chain and tree kernels
 *    give that row out_count[b] = -1 (its other outputs are then unspecified), and
 *    spec_verify_rows_status turns it into the call's SV_ERR_TIMEOUT.  The
 *    position-parallel small-batch chain kernel reports such a row as invalid data
 *    (out_count[b] = 0): its per-row word has no room for a third state.
 *  - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* a size, pointer, dtype or kind argument is invalid */
    SV_ERR_UNSUPPORTED = 2, /* valid but outside what the library handles (size limits, device) */
    SV_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    SV_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up on some row (out_count = -1, see
                               spec_verify_rows_status); re-zero the workspace before reusing it */
    SV_ERR_BAD_INPUT = 5    /* some batch rows held invalid data (see spec_verify_count_invalid) */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum { SV_DRAFT_PROBS = 0, SV_DRAFT_LOGITS = 1 } sv_draft_kind;

/*
 * Bytes of device workspace spec_verify_chain may use for B batch rows, K drafts
 * and vocabulary V.  The caller zero-fills the workspace once before its first
 * use; every successful call leaves it zeroed again.  Passing a smaller (or NULL)
 * workspace is allowed and selects a path that needs none.
 */
SV_API size_t spec_verify_workspace_size(int B, int K, int V);

/*
 * Chain verify (sampling and greedy rows mixed by temperature).
 *   target_logits  device [B][K+1][V], dtype tdt.  Row k is the target's next-token
 *                  logits at chain position k (k = K: the bonus position).
 *   draft          device [B][K][V]: SV_DRAFT_PROBS -> fp32 probabilities q_k;
 *                  SV_DRAFT_LOGITS -> logits of dtype ddt, q_k = softmax(row / T).
 *                  Not read for greedy rows; required (non-NULL) when K > 0.
 *   draft_tokens   device int32 [B][K], the drafted tokens x_0..x_{K-1}.
 *   temperature    device fp32 [B].
 *   B >= 0, 0 <= K <= 64, 1 <= V <= 1<<24.
 *   seed, offset   Philox key word and counter word (see conventions).
 *   out_tokens     device int32 [B][K+1]: accepted drafts, then the replacement or
 *                  bonus token; unused slots are -1.
 *   out_count      device int32 [B]: number of valid entries in out_tokens[b]
 *                  (1..K+1; 0 for an invalid row; -1 where a bounded wait gave up).
 *   out_accept_prob  nullable device fp32 [B][K]: min(1, p_k(x_k)/q_k(x_k)) for every
 *                  position up to and including the first rejection (greedy rows:
 *                  1 for a match, 0 for the mismatch); -1 for positions never
 *                  evaluated.
 *   workspace, ws_bytes  optional scratch (see spec_verify_workspace_size).
 * Rows after the first rejection never affect the result and are not validated
 * (invalid data there leaves the row valid).  With a workspace, small and moderate
 * batches run a kernel that reads every position at once to shorten the critical
 * path; the other kernels stop reading at the first rejection.
 */
SV_API sv_status spec_verify_chain(const void *target_logits, sv_dtype tdt,
                            const void *draft, sv_dtype ddt, sv_draft_kind dk,
                            const int32_t *draft_tokens, const float *temperature,
                            int B, int K, int V, uint64_t seed, uint64_t offset,
                            int32_t *out_tokens, int32_t *out_count, float *out_accept_prob,
                            void *workspace, size_t ws_bytes, void *stream);

/*
 * Chain verify that allocates nothing (the pages have no counterpart: this is a
 * deployment convenience).  For callers that cannot hand the library a workspace:
 * code running inside a runtime that owns every device allocation (an engine's
 * memory arena, a plugin interface that passes only input and output buffers) or a
 * path on which no allocation call is allowed.  Same arguments and outputs as
 * spec_verify_chain, minus the workspace, and the same kernel choice: where
 * spec_verify_chain would run the position-parallel kernel (small and moderate
 * batches, aligned rows) this entry runs it too, with its scratch in a 256 KiB array
 * inside the library's device image, present on every device that loads the library
 * until the process exits; elsewhere it runs the kernels that need no scratch.
 * Results agree with spec_verify_chain except where a decision lies within fp32
 * rounding of its boundary.  No cudaMalloc, cudaFree or other allocating call is made.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and zeroes it synchronously;
 *     make that first call before any stream capture.
 *   - Calls whose scratch would exceed 256 KiB (spec_verify_workspace_size(B, K, V) >
 *     256 KiB) return SV_ERR_UNSUPPORTED without launching anything.
 *   - Every call shares the one array: calls that overlap on the GPU (different
 *     streams, or different host threads) race and must be serialised by the caller.
 */
SV_API sv_status spec_verify_chain_noalloc(const void *target_logits, sv_dtype tdt,
                                    const void *draft, sv_dtype ddt, sv_draft_kind dk,
                                    const int32_t *draft_tokens, const float *temperature,
                                    int B, int K, int V, uint64_t seed, uint64_t offset,
                                    int32_t *out_tokens, int32_t *out_count, float *out_accept_prob,
                                    void *stream);

/*
 * Chain verify from host memory (the pages have no counterpart: this is the serving
 * loop's round trip).  One call enqueues on `stream`, without synchronising:
 *   1. one host-to-device copy of a round's packed inputs, h_in -> d_in;
 *   2. spec_verify_chain on views of d_in, writing into d_out;
 *   3. one device-to-host copy of the outputs, d_out -> h_out.
 * The packed input layout, each part starting at a multiple of 256 bytes:
 *   target [B][K+1][V] (tdt), draft [B][K][V] (ddt, fp32 for SV_DRAFT_PROBS),
 *   tokens int32 [B][K], temperature fp32 [B].
 * The packed output layout: tokens int32 [B][K+1], then counts int32 [B].
 *   h_in, h_out    host buffers; page-locked (pinned) for the copies to be asynchronous.
 *   d_in, d_out    device buffers of in_bytes and out_bytes (spec_verify_host_sizes).
 *   workspace, ws_bytes  as spec_verify_chain.
 * The outputs in h_out are valid once the stream has reached this call's end (an event
 * or a synchronisation).  Independent rounds on several streams in turn, each stream
 * with its own d_in / d_out pair and workspace, overlap one round's copy with the
 * verifies (and the copies' fixed start-up latency) of the rounds before it.  Errors: those of
 * spec_verify_chain; SV_ERR_INVALID_ARG for a NULL buffer; SV_ERR_CUDA when a copy cannot
 * be enqueued.
 */
SV_API sv_status spec_verify_chain_host(const void *h_in, void *d_in, void *h_out, void *d_out,
                                        sv_dtype tdt, sv_dtype ddt, sv_draft_kind dk, int B, int K, int V,
                                        uint64_t seed, uint64_t offset, void *workspace, size_t ws_bytes,
                                        void *stream);

/*
 * Sizes of spec_verify_chain_host's packed buffers.  offsets (nullable) receives 4
 * byte offsets into the packed input: target, draft, tokens, temperature.  Returns
 * SV_ERR_INVALID_ARG for sizes outside spec_verify_chain's limits or an unknown dtype
 * or kind.
 */
SV_API sv_status spec_verify_host_sizes(int B, int K, int V, sv_dtype tdt, sv_dtype ddt, sv_draft_kind dk,
                                        size_t *offsets, size_t *in_bytes, size_t *out_bytes);

/*
 * Greedy acceptance (the temperature-0 rule) for every row:
 *   target_logits device [B][K+1][V] (tdt), draft_tokens device int32 [B][K];
 *   out_tokens device int32 [B][K+1], out_count device int32 [B].
 * Accepts x_k while x_k == argmax(row k); emits argmax of the first mismatching row
 * (or of row K when all match).  No draft distribution is read.
 */
SV_API sv_status spec_greedy_accept(const void *target_logits, sv_dtype tdt, const int32_t *draft_tokens,
                             int B, int K, int V, int32_t *out_tokens, int32_t *out_count,
                             void *stream);

/*
 * Tree verify.
 *   target_logits  device [B][N+1][V] (tdt): row 0 is the root's next-token logits,
 *                  row i+1 the next-token logits after node i.
 *   draft          device [B][N+1][V], the same row layout (probs fp32 or logits ddt);
 *                  row r is the draft distribution the children of that row's node
 *                  were proposed from.  Not read for greedy rows.
 *   node_tokens    device int32 [B][N]; parent device int32 [B][N] with parent[i] in
 *                  {-1} u [0, i) (-1: child of the root).  Children of a node are tried
 *                  in increasing node index.
 *   temperature    device fp32 [B].  1 <= N <= 1024, 1 <= max_depth <= 64, max_depth at
 *                  least the depth of every node (else the row is invalid).
 *   out_tokens     device int32 [B][max_depth+1]: the accepted node tokens along the
 *                  path, then the final drawn (or argmax) token; -1 padded.
 *   out_count      device int32 [B] (1..depth+1; 0 for an invalid row).
 *   out_path       device int32 [B][max_depth]: accepted node indices, -1 padded.
 * Greedy rows descend into the lowest-index child whose token equals the argmax of
 * the current row.  Sampling rows try the children in order with acceptance
 * r < p(x)/q(x); after a rejection p <- (p - q)+ / |(p - q)+|_1 (kept if that mass
 * is zero), q(x) <- 0 and q is renormalised.  With no child accepted, or at a
 * leaf, the last token is drawn from the current p.
 */
SV_API sv_status spec_verify_tree(const void *target_logits, sv_dtype tdt,
                           const void *draft, sv_dtype ddt, sv_draft_kind dk,
                           const int32_t *node_tokens, const int32_t *parent,
                           const float *temperature, int B, int N, int V, int max_depth,
                           uint64_t seed, uint64_t offset,
                           int32_t *out_tokens, int32_t *out_count, int32_t *out_path,
                           void *stream);

/*
 * Draft sampling and verify in one call, for drafters whose K next-token
 * distributions are all known up front (several prediction heads on one hidden
 * state): x_k is drawn from q_k = softmax(draft_logits_k / T) ("[논문 리뷰] Fast
 * Inference from Transformers via Speculative Decoding", section 2, Step 1: the
 * draft proposes by sampling from its own distribution), then the K tokens are
 * verified exactly as spec_verify_chain does with the draft given as logits.
 *   draft_logits   device [B][K][V] (ddt); the same array q is computed from in the verify.
 *   out_draft_tokens device int32 [B][K]: the drafted tokens (-1 where a draft row is
 *                  invalid data, which makes that batch row invalid: count 0).
 * x_k is the inverse-CDF draw of word 2 of Philox slot k (words 0 and 1 keep their
 * roles), on the same 24-bit grid; a greedy row (T <= 0) drafts x_k = argmax of
 * draft row k (lowest index on ties) and is verified greedily.  Other arguments,
 * outputs, workspace use and errors as spec_verify_chain.  Two kernels run on
 * `stream`: the sampling kernel, then the verify kernel.
 */
SV_API sv_status spec_sample_and_verify(const void *target_logits, sv_dtype tdt,
                                        const void *draft_logits, sv_dtype ddt,
                                        const float *temperature, int B, int K, int V,
                                        uint64_t seed, uint64_t offset, int32_t *out_draft_tokens,
                                        int32_t *out_tokens, int32_t *out_count, float *out_accept_prob,
                                        void *workspace, size_t ws_bytes, void *stream);

/*
 * How the children of one node were drafted, which decides what a rejection does
 * to the draft distribution before the next sibling is tried ("Progressive Tree
 * Drafting" summary, section "검증": sampling acceptance without replacement;
 * drafts sampled independently from q are the multi-draft case of the same rule).
 *  SV_SIBLINGS_WITHOUT_REPLACEMENT: the children are distinct tokens drawn without
 *    replacement from q; after rejecting token x, q(x) <- 0 and q is renormalised.
 *  SV_SIBLINGS_IID: the children were drawn independently from q (a token may
 *    repeat); q is left as it is.
 * Both set p <- (p - q)+ / |(p - q)+|_1 after a rejection, and both give outputs
 * distributed exactly as the target when the children were drafted that way.
 */
typedef enum { SV_SIBLINGS_WITHOUT_REPLACEMENT = 0, SV_SIBLINGS_IID = 1 } sv_sibling_rule;

/* spec_verify_tree with an explicit sibling rule (spec_verify_tree uses
 * SV_SIBLINGS_WITHOUT_REPLACEMENT).  Same arguments, outputs and errors, plus
 * SV_ERR_INVALID_ARG for an unknown rule. */
SV_API sv_status spec_verify_tree_rule(const void *target_logits, sv_dtype tdt,
                                       const void *draft, sv_dtype ddt, sv_draft_kind dk,
                                       const int32_t *node_tokens, const int32_t *parent,
                                       const float *temperature, int B, int N, int V, int max_depth,
                                       sv_sibling_rule sibling_rule, uint64_t seed, uint64_t offset,
                                       int32_t *out_tokens, int32_t *out_count, int32_t *out_path,
                                       void *stream);

/* Static, NUL-terminated description of a status code. */
SV_API const char *spec_verify_status_string(sv_status status);

/* Description of the CUDA error behind the most recent SV_ERR_CUDA returned on the
 * calling thread ("no CUDA error" if there was none).  Static storage; not freed. */
SV_API const char *spec_verify_last_cuda_error(void);

/*
 * Data-error status of a finished verify call.  The verify entries report bad data
 * per batch row, as out_count[b] = 0 (NaN or +inf in a row the rule read, a row with
 * no finite logit, an out-of-range token, a malformed tree), and still process the
 * other rows; they return SV_OK for such calls.  This counts those rows on the
 * device, in stream order after the call: a non-zero count is the call's
 * SV_ERR_BAD_INPUT, and the rows are the ones whose count is 0.
 *   out_count    device int32 [B], as written by spec_verify_chain(_noalloc),
 *                spec_greedy_accept, spec_verify_tree(_rule) or spec_sample_and_verify.
 *   B            0 <= B <= 1<<24.
 *   out_invalid  device int32, written once (no initialisation needed).
 * One kernel on `stream`; nothing is allocated.  Errors: SV_ERR_INVALID_ARG (B out of
 * range, out_invalid NULL, out_count NULL with B > 0), SV_ERR_CUDA (launch failure).
 */
SV_API sv_status spec_verify_count_invalid(const int32_t *out_count, int B, int32_t *out_invalid, void *stream);

/*
 * Row status of a finished verify call (the pages have no counterpart: this reports
 * device-side failures).  Rows with out_count[b] = -1 are rows on which a bounded
 * device-side wait gave up; rows with out_count[b] = 0 hold invalid data.
 * Writes, on the device and in stream order after the call:
 *   out_status[0]  the call's status: SV_ERR_TIMEOUT if any row has count -1, else
 *                  SV_ERR_BAD_INPUT if any row has count 0, else SV_OK;
 *   out_status[1]  the number of rows with count 0;
 *   out_status[2]  the number of rows with count -1.
 *   out_count    device int32 [B], as any verify entry writes it; 0 <= B <= 1<<24.
 *   out_status   device int32 [3], written once (no initialisation needed).
 * One kernel on `stream`; nothing is allocated.  Errors: SV_ERR_INVALID_ARG (B out of
 * range, out_status NULL, out_count NULL with B > 0), SV_ERR_CUDA (launch failure).
 */
SV_API sv_status spec_verify_rows_status(const int32_t *out_count, int B, int32_t *out_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
