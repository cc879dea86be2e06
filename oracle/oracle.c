/*
 * oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, single-threaded fp64 restatement of the target-side
 * verify/accept step of speculative decoding.  Only tests/,
 * __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg load it.
 * It shares no code, header, table or constant with the CUDA library: the
 * Philox generator, the bf16 widening and every step below are written here
 * independently.
 *
 * Sources (page title, section):
 *  - "[논문 리뷰] Fast Inference from Transformers via Speculative Decoding"
 *    (velog review of Leviathan et al., ICML 2023), section 2 "제안 방법":
 *    left-to-right acceptance with probability min(1, p(x)/q(x)); on the
 *    first rejection resample from max(0, p-q)/sum max(0, p-q); one bonus
 *    token when all K pass; 1..K+1 tokens per round.
 *  - "Speculative Decoding and EAGLE" (pai-world lesson), section
 *    "정확성 규칙 (The Exactness Rule)": r ~ U(0,1), accept iff r < p/q,
 *    residual (p-q)+/||(p-q)+||_1; greedy case: accept iff argmax(p) == x_t,
 *    else emit argmax(p) and stop.  Same page, section "개념": a bonus token
 *    from p(. | x_1..x_K) when every draft passes.
 *  - "Progressive Tree Drafting" summary (gist.science, arXiv 2607.10661),
 *    section "검증 (Verification)": greedy tree acceptance (an edge is
 *    accepted when the verified token equals a child) and sampling tree
 *    acceptance without replacement from normalised probabilities.  The exact
 *    sibling rule used here (siblings in index order; on reject
 *    p <- norm((p-q)+), the tried token zeroed in q, q renormalised) is the
 *    tree workload's stated rule.
 *
 * Readings where the pages are silent (stated once, used throughout):
 *  - temperature: p = softmax(l / T); T <= 0 (or NaN) selects greedy.  A draft
 *    given as logits uses the same T; a draft given as probabilities is used
 *    as given.
 *  - random numbers: Philox4x64-10 (Salmon et al., SC'11), counter
 *    {slot, row, offset, 0}, key {seed, 0}.  Word 0 of slot k is the accept
 *    uniform of position k (tree: of node k); word 1 of slot k is the draw
 *    uniform at position k (tree: at distribution row k).  A uniform is
 *    (w >> 40) * 2^-24, a 24-bit grid in [0, 1).
 *  - q(x) == 0: accept iff p(x) > 0.  Ties in argmax: lowest index.
 *  - residual with zero mass: draw from p instead.
 *  - greedy bonus: argmax of the last row.
 *  - invalid data (a read row containing NaN or +inf, or all -inf; a token
 *    outside [0, V); a malformed parent array; a draft probability at the
 *    drafted token that is negative or not finite) gives count 0 and all
 *    output slots -1.
 *  - margins: every sampled decision records |r - ratio|; every draw records
 *    the distance from t = u * Z to the nearest CDF boundary, in probability
 *    mass.  The minimum over a row is returned so that a parity check can
 *    excuse rows an fp32 implementation may legitimately decide differently.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_DRAFT_PROBS 0
#define ORC_DRAFT_LOGITS 1

/* ---------------------------------------------------------------- Philox */

static void orc_mul128(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    unsigned __int128 prod = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(prod >> 64);
    *lo = (uint64_t)prod;
}

/* Philox4x64 with 10 rounds: each round multiplies counter words 0 and 2 by
 * the two round multipliers, swaps the halves and xors in the key; the key is
 * bumped by the two Weyl constants between rounds. */
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t mul_a = 0xD2E7470EE14C6C93ULL, mul_b = 0xCA5A826395121157ULL;
    const uint64_t weyl_a = 0x9E3779B97F4A7C15ULL, weyl_b = 0xBB67AE8584CAA73BULL;
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t hi_a, lo_a, hi_b, lo_b;
        orc_mul128(mul_a, x0, &hi_a, &lo_a);
        orc_mul128(mul_b, x2, &hi_b, &lo_b);
        uint64_t y0 = hi_b ^ x1 ^ k0;
        uint64_t y1 = lo_b;
        uint64_t y2 = hi_a ^ x3 ^ k1;
        uint64_t y3 = lo_a;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += weyl_a;
        k1 += weyl_b;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

static double orc_u24(uint64_t w) { return (double)(w >> 40) * (1.0 / 16777216.0); }

/* Both uniforms of one slot: *r from word 0, *u from word 1. */
static void orc_slot_uniforms(uint64_t seed, uint64_t offset, uint64_t row, uint64_t slot,
                              double *r, double *u)
{
    uint64_t c[4] = {slot, row, offset, 0}, k[2] = {seed, 0}, w[4];
    oracle_philox4x64_10(c, k, w);
    *r = orc_u24(w[0]);
    *u = orc_u24(w[1]);
}

/* ------------------------------------------------------------ elements */

static double orc_load(const void *base, int dt, size_t idx)
{
    if (dt == ORC_F32) return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16; /* bf16 = top half of f32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Maximum of a row; returns 0 when the row is valid (no NaN, no +inf, not all -inf). */
static int orc_row_max(const void *base, int dt, size_t off, int V, double *m_out, int *argmax_out)
{
    double m = -INFINITY;
    int am = -1;
    for (int i = 0; i < V; ++i) {
        double x = orc_load(base, dt, off + (size_t)i);
        if (isnan(x) || x == INFINITY) return -1;
        if (x > m) { m = x; am = i; }
    }
    if (m == -INFINITY) return -1;
    *m_out = m;
    if (argmax_out) *argmax_out = am;
    return 0;
}

/* Temperature softmax of one row: p_i = exp((l_i - max)/T) / sum_j exp((l_j - max)/T). */
static int orc_softmax(const void *base, int dt, size_t off, int V, double T, double *p)
{
    double m;
    if (orc_row_max(base, dt, off, V, &m, NULL)) return -1;
    double S = 0.0;
    for (int i = 0; i < V; ++i) {
        double e = exp((orc_load(base, dt, off + (size_t)i) - m) / T);
        p[i] = e;
        S += e;
    }
    for (int i = 0; i < V; ++i) p[i] /= S;
    return 0;
}

/* Inverse-CDF draw: Z = sum w (index order), t = u * Z, the token is the smallest i
 * with C_i > t where C_i = w_0 + ... + w_i.  *margin gets min(t - C_{i-1}, C_i - t). */
static int orc_draw(const double *w, int V, double u, double *margin)
{
    double Z = 0.0;
    for (int i = 0; i < V; ++i) Z += w[i];
    double t = u * Z, C = 0.0;
    int last_nonzero = -1;
    for (int i = 0; i < V; ++i) {
        double Cn = C + w[i];
        if (w[i] > 0.0) last_nonzero = i;
        if (Cn > t) {
            double a = t - C, b = Cn - t;
            *margin = a < b ? a : b;
            return i;
        }
        C = Cn;
    }
    *margin = 0.0; /* unreachable for u < 1 and Z > 0 */
    return last_nonzero;
}

/* Acceptance ratio p/q with the q == 0 reading (accept iff p > 0). */
static double orc_ratio(double px, double qx)
{
    if (qx > 0.0) return px / qx;
    return px > 0.0 ? INFINITY : 0.0;
}

static double orc_min(double a, double b) { return a < b ? a : b; }

/* ------------------------------------------------------------- chain */

/*
 * Chain verify with explicit uniforms.
 *  target  [B][K+1][V] (f32 or bf16), draft [B][K][V] (probs f32, or logits f32/bf16),
 *  tokens  [B][K], temperature [B], r [B][K] accept uniforms, u [B][K+1] draw uniforms.
 * Outputs: out_tokens [B][K+1] (-1 padded), out_count [B], out_accept_prob [B][K]
 * (min(1,p/q) for evaluated positions, greedy: 1/0; -1 elsewhere; nullable),
 * out_margin [B] (nullable; +inf when no sampled decision was taken).
 * Returns the number of invalid rows.
 */
int oracle_verify_chain_u(const void *target, int tdt, const void *draft, int ddt, int dk,
                          const int32_t *tokens, const float *temperature, int B, int K, int V,
                          const double *r, const double *u, int32_t *out_tokens,
                          int32_t *out_count, float *out_accept_prob, double *out_margin)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    int n_invalid = 0;
    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * (K + 1);
        float *ap = out_accept_prob ? out_accept_prob + (size_t)b * K : NULL;
        for (int k = 0; k <= K; ++k) ot[k] = -1;
        if (ap) for (int k = 0; k < K; ++k) ap[k] = -1.0f;
        double margin = INFINITY;
        int emitted = 0, invalid = 0;
        const int32_t *x = tokens + (size_t)b * K;
        for (int k = 0; k < K; ++k)
            if (x[k] < 0 || x[k] >= V) invalid = 1;
        double T = (double)temperature[b];
        int greedy = !(T > 0.0);
        for (int k = 0; k <= K && !invalid; ++k) {
            size_t toff = ((size_t)b * (K + 1) + k) * (size_t)V;
            if (greedy) {
                double m;
                int g;
                if (orc_row_max(target, tdt, toff, V, &m, &g)) { invalid = 1; break; }
                if (k < K && x[k] == g) {
                    ot[emitted++] = x[k];
                    if (ap) ap[k] = 1.0f;
                    continue;
                }
                if (k < K && ap) ap[k] = 0.0f;
                ot[emitted++] = g;
                break;
            }
            if (orc_softmax(target, tdt, toff, V, T, p)) { invalid = 1; break; }
            if (k == K) { /* every draft accepted: bonus token from p at position K */
                double mg;
                ot[emitted++] = orc_draw(p, V, u[(size_t)b * (K + 1) + K], &mg);
                margin = orc_min(margin, mg);
                break;
            }
            size_t doff = ((size_t)b * K + k) * (size_t)V;
            if (dk == ORC_DRAFT_LOGITS) {
                if (orc_softmax(draft, ddt, doff, V, T, q)) { invalid = 1; break; }
            } else {
                for (int i = 0; i < V; ++i) q[i] = orc_load(draft, ORC_F32, doff + (size_t)i);
                if (!(q[x[k]] >= 0.0) || !isfinite(q[x[k]])) { invalid = 1; break; }
            }
            double ratio = orc_ratio(p[x[k]], q[x[k]]);
            double rk = r[(size_t)b * K + k];
            if (ap) ap[k] = (float)(ratio < 1.0 ? ratio : 1.0);
            margin = orc_min(margin, fabs(rk - ratio));
            if (rk < ratio) { ot[emitted++] = x[k]; continue; }
            /* first rejection: replacement from the residual (p - q)+ */
            double Z = 0.0;
            for (int i = 0; i < V; ++i) {
                double d = p[i] - q[i];
                w[i] = d > 0.0 ? d : 0.0;
                Z += w[i];
            }
            if (!(Z > 0.0)) memcpy(w, p, sizeof(double) * (size_t)V);
            double mg;
            ot[emitted++] = orc_draw(w, V, u[(size_t)b * (K + 1) + k], &mg);
            margin = orc_min(margin, mg);
            break;
        }
        if (invalid) {
            for (int k = 0; k <= K; ++k) ot[k] = -1;
            if (ap) for (int k = 0; k < K; ++k) ap[k] = -1.0f;
            emitted = 0;
            ++n_invalid;
        }
        out_count[b] = emitted;
        if (out_margin) out_margin[b] = margin;
    }
    free(p);
    free(q);
    free(w);
    return n_invalid;
}

/* Chain verify with the Philox stream; row_id (nullable) maps local row b to the
 * row index used in the counter, so that a subset of a batch can be recomputed. */
int oracle_verify_chain(const void *target, int tdt, const void *draft, int ddt, int dk,
                        const int32_t *tokens, const float *temperature, int B, int K, int V,
                        uint64_t seed, uint64_t offset, const int32_t *row_id,
                        int32_t *out_tokens, int32_t *out_count, float *out_accept_prob,
                        double *out_margin)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)B * (K > 0 ? K : 1));
    double *u = (double *)malloc(sizeof(double) * (size_t)B * (K + 1));
    for (int b = 0; b < B; ++b) {
        uint64_t rid = row_id ? (uint64_t)row_id[b] : (uint64_t)b;
        for (int k = 0; k <= K; ++k) {
            double rr, uu;
            orc_slot_uniforms(seed, offset, rid, (uint64_t)k, &rr, &uu);
            if (k < K) r[(size_t)b * K + k] = rr;
            u[(size_t)b * (K + 1) + k] = uu;
        }
    }
    int n = oracle_verify_chain_u(target, tdt, draft, ddt, dk, tokens, temperature, B, K, V, r, u,
                                  out_tokens, out_count, out_accept_prob, out_margin);
    free(r);
    free(u);
    return n;
}

/* Greedy acceptance only: every row uses argmax acceptance (temperature 0). */
int oracle_greedy_accept(const void *target, int tdt, const int32_t *tokens, int B, int K, int V,
                         int32_t *out_tokens, int32_t *out_count)
{
    float *temps = (float *)calloc((size_t)(B > 0 ? B : 1), sizeof(float));
    int n = oracle_verify_chain_u(target, tdt, NULL, ORC_F32, ORC_DRAFT_PROBS, tokens, temps, B, K, V,
                                  NULL, NULL, out_tokens, out_count, NULL, NULL);
    free(temps);
    return n;
}

/* -------------------------------------------------------------- tree */

/*
 * Tree verify with explicit uniforms.
 *  target/draft [B][N+1][V]: row 0 is the root's next-token distribution, row i+1
 *  the distribution after node i.  node_tokens/parent [B][N] with parent[i] in
 *  {-1} u [0, i).  r [B][N]: accept uniform of node i.  u [B][N+1]: draw uniform at
 *  row i.  Outputs: out_tokens [B][D+1], out_count [B], out_path [B][D] (accepted
 *  node indices), out_margin [B] (nullable).  Returns the number of invalid rows.
 *  sibling_rule: ORC_SIBLINGS_WOR (0), siblings drafted without replacement: a
 *  rejected token's draft probability is zeroed and q renormalised; ORC_SIBLINGS_IID
 *  (1), siblings drafted i.i.d. from q: q is left as it is (the multi-draft rule of
 *  SpecInfer-style verifiers; "Progressive Tree Drafting", section "검증", names the
 *  without-replacement case).  Both keep p <- norm((p - q)+) after a rejection.
 */
#define ORC_SIBLINGS_WOR 0
#define ORC_SIBLINGS_IID 1
int oracle_verify_tree_rule_u(const void *target, int tdt, const void *draft, int ddt, int dk,
                              const int32_t *node_tokens, const int32_t *parent,
                              const float *temperature, int B, int N, int V, int max_depth,
                              int sibling_rule, const double *r, const double *u, int32_t *out_tokens,
                              int32_t *out_count, int32_t *out_path, double *out_margin)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *wn = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    int *depth = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    int n_invalid = 0;
    const int D = max_depth;
    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * (D + 1);
        int32_t *op = out_path + (size_t)b * (D > 0 ? D : 0);
        for (int i = 0; i <= D; ++i) ot[i] = -1;
        for (int i = 0; i < D; ++i) op[i] = -1;
        const int32_t *tok = node_tokens + (size_t)b * N;
        const int32_t *par = parent + (size_t)b * N;
        int invalid = 0;
        for (int i = 0; i < N; ++i) {
            if (tok[i] < 0 || tok[i] >= V) invalid = 1;
            if (par[i] < -1 || par[i] >= i) { invalid = 1; depth[i] = 0; continue; }
            depth[i] = par[i] < 0 ? 1 : depth[par[i]] + 1;
            if (depth[i] > D) invalid = 1;
        }
        double T = (double)temperature[b];
        int greedy = !(T > 0.0);
        double margin = INFINITY;
        int emitted = 0, cur = -1;
        while (!invalid) {
            int row = cur + 1;
            size_t off = ((size_t)b * (N + 1) + row) * (size_t)V;
            if (greedy) {
                double m;
                int g;
                if (orc_row_max(target, tdt, off, V, &m, &g)) { invalid = 1; break; }
                int next = -1;
                for (int c = 0; c < N; ++c)
                    if (par[c] == cur && tok[c] == g) { next = c; break; }
                ot[emitted] = g;
                if (next < 0) { ++emitted; break; }
                op[emitted++] = next;
                cur = next;
                continue;
            }
            /* current distribution p = w / Zl; level 0 is the softmax itself (Zl = 1) */
            if (orc_softmax(target, tdt, off, V, T, w)) { invalid = 1; break; }
            double Zl = 1.0;
            int have_q = 0, next = -1;
            for (int c = 0; c < N && next < 0; ++c) {
                if (par[c] != cur) continue;
                if (!have_q) {
                    if (dk == ORC_DRAFT_LOGITS) {
                        if (orc_softmax(draft, ddt, off, V, T, q)) { invalid = 1; break; }
                    } else {
                        for (int i = 0; i < V; ++i) q[i] = orc_load(draft, ORC_F32, off + (size_t)i);
                    }
                    have_q = 1;
                }
                int x = tok[c];
                if (dk == ORC_DRAFT_PROBS && (!(q[x] >= 0.0) || !isfinite(q[x]))) { invalid = 1; break; }
                double ratio = orc_ratio(w[x] / Zl, q[x]);
                double rc = r[(size_t)b * N + c];
                margin = orc_min(margin, fabs(rc - ratio));
                if (rc < ratio) { next = c; break; }
                /* sibling rejected: p <- norm((p - q)+); without replacement also q[x] <- 0, q <- norm(q) */
                double Zn = 0.0;
                for (int i = 0; i < V; ++i) {
                    double d = w[i] / Zl - q[i];
                    wn[i] = d > 0.0 ? d : 0.0;
                    Zn += wn[i];
                }
                if (Zn > 0.0) {
                    memcpy(w, wn, sizeof(double) * (size_t)V);
                    Zl = Zn;
                }
                if (sibling_rule == ORC_SIBLINGS_IID) continue;
                q[x] = 0.0;
                double Sq = 0.0;
                for (int i = 0; i < V; ++i) Sq += q[i];
                if (Sq > 0.0)
                    for (int i = 0; i < V; ++i) q[i] /= Sq;
            }
            if (invalid) break;
            if (next >= 0) {
                ot[emitted] = tok[next];
                op[emitted++] = next;
                cur = next;
                continue;
            }
            double mg;
            ot[emitted++] = orc_draw(w, V, u[(size_t)b * (N + 1) + row], &mg);
            margin = orc_min(margin, mg);
            break;
        }
        if (invalid) {
            for (int i = 0; i <= D; ++i) ot[i] = -1;
            for (int i = 0; i < D; ++i) op[i] = -1;
            emitted = 0;
            ++n_invalid;
        }
        out_count[b] = emitted;
        if (out_margin) out_margin[b] = margin;
    }
    free(w);
    free(wn);
    free(q);
    free(depth);
    return n_invalid;
}

int oracle_verify_tree_u(const void *target, int tdt, const void *draft, int ddt, int dk,
                         const int32_t *node_tokens, const int32_t *parent,
                         const float *temperature, int B, int N, int V, int max_depth,
                         const double *r, const double *u, int32_t *out_tokens,
                         int32_t *out_count, int32_t *out_path, double *out_margin)
{
    return oracle_verify_tree_rule_u(target, tdt, draft, ddt, dk, node_tokens, parent, temperature, B, N, V,
                                     max_depth, ORC_SIBLINGS_WOR, r, u, out_tokens, out_count, out_path,
                                     out_margin);
}

/* Tree verify with the Philox stream (same slot layout as the chain, so a tree whose
 * parent array is a chain reproduces the chain's outputs). */
int oracle_verify_tree_rule(const void *target, int tdt, const void *draft, int ddt, int dk,
                            const int32_t *node_tokens, const int32_t *parent, const float *temperature,
                            int B, int N, int V, int max_depth, int sibling_rule, uint64_t seed,
                            uint64_t offset, const int32_t *row_id, int32_t *out_tokens, int32_t *out_count,
                            int32_t *out_path, double *out_margin)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)B * (N > 0 ? N : 1));
    double *u = (double *)malloc(sizeof(double) * (size_t)B * (N + 1));
    for (int b = 0; b < B; ++b) {
        uint64_t rid = row_id ? (uint64_t)row_id[b] : (uint64_t)b;
        for (int s = 0; s <= N; ++s) {
            double rr, uu;
            orc_slot_uniforms(seed, offset, rid, (uint64_t)s, &rr, &uu);
            if (s < N) r[(size_t)b * N + s] = rr;
            u[(size_t)b * (N + 1) + s] = uu;
        }
    }
    int n = oracle_verify_tree_rule_u(target, tdt, draft, ddt, dk, node_tokens, parent, temperature, B, N,
                                      V, max_depth, sibling_rule, r, u, out_tokens, out_count, out_path,
                                      out_margin);
    free(r);
    free(u);
    return n;
}

int oracle_verify_tree(const void *target, int tdt, const void *draft, int ddt, int dk,
                       const int32_t *node_tokens, const int32_t *parent, const float *temperature,
                       int B, int N, int V, int max_depth, uint64_t seed, uint64_t offset,
                       const int32_t *row_id, int32_t *out_tokens, int32_t *out_count,
                       int32_t *out_path, double *out_margin)
{
    return oracle_verify_tree_rule(target, tdt, draft, ddt, dk, node_tokens, parent, temperature, B, N, V,
                                   max_depth, ORC_SIBLINGS_WOR, seed, offset, row_id, out_tokens, out_count,
                                   out_path, out_margin);
}

/* ------------------------------------------------------ tree attention mask */

/*
 * Ancestor-or-self mask of a draft tree ("Speculative Decoding and EAGLE", section
 * "트리 어텐션 검증": each node attends only to its ancestors in the tree; the node
 * itself is included, as causal attention always includes the current token;
 * "Progressive Tree Drafting", section "트리 구조 드래프팅": the attention mask is
 * rebuilt so one forward pass follows every branch).
 *  parent [B][N] with parent[i] in {-1} u [0, i).  mask [B][N][W], W = (N+31)/32,
 *  bit j of row i set iff j is i or an ancestor of i.  depth [B][N]: nodes on the
 *  path from the root's child down to i (1 for a child of the root).  valid [B]:
 *  1, or 0 for a malformed parent array (its mask rows and depths are then 0).
 */
int oracle_tree_mask(const int32_t *parent, int B, int N, uint32_t *mask, int32_t *depth, int32_t *valid)
{
    const int W = (N + 31) / 32;
    int n_invalid = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        uint32_t *m = mask + (size_t)b * N * W;
        int32_t *dp = depth + (size_t)b * N;
        int ok = 1;
        for (int i = 0; i < N; ++i)
            if (par[i] < -1 || par[i] >= i) ok = 0;
        memset(m, 0, sizeof(uint32_t) * (size_t)N * W);
        for (int i = 0; i < N; ++i) dp[i] = 0;
        if (ok) {
            for (int i = 0; i < N; ++i) {
                int d = 0;
                for (int j = i; j >= 0; j = par[j]) {  /* walk up to the root */
                    m[(size_t)i * W + j / 32] |= 1u << (j % 32);
                    ++d;
                }
                dp[i] = d;
            }
        } else {
            ++n_invalid;
        }
        valid[b] = ok;
    }
    return n_invalid;
}

/* --------------------------------------------------- accepted-path KV compaction */

/*
 * KV-cache rollback after a tree verify (the velog review of Leviathan et al.,
 * section 4 "한계점": the KV entries of rejected tokens must be rolled back).  Tree
 * node i's cache row sits at base[b] + i; the accepted nodes path[0..L-1]
 * (L = count - 1: the last emitted token has no cache row yet) are moved, in order,
 * to rows base[b] + 0..L-1: for d = 0..L-1, row base+d <- row base+path[d].
 * kv: bytes, row r of batch row b at b*batch_stride + r*row_stride, row_bytes each.
 * A batch row whose count is 0 or above D + 1, whose path has an entry path[d] < d,
 * or whose rows fall outside [0, num_rows) is left untouched.  (With path[d] >= d no
 * step reads a row an earlier step wrote, so the in-order copy equals a gather from
 * the cache as it was before the call.)
 */
int oracle_kv_compact(unsigned char *kv, size_t batch_stride, size_t row_stride, size_t row_bytes,
                      const int32_t *path, const int32_t *count, const int32_t *base, int B, int D, int num_rows)
{
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *pth = path + (size_t)b * D;
        const int L = count[b] - 1;
        int ok = count[b] >= 1 && L <= D;
        for (int d = 0; ok && d < L; ++d)
            if (pth[d] < d || base[b] < 0 || base[b] + pth[d] >= num_rows) ok = 0;
        if (!ok) { ++skipped; continue; }
        unsigned char *rowb = kv + (size_t)b * batch_stride;
        for (int d = 0; d < L; ++d)
            memmove(rowb + (size_t)(base[b] + d) * row_stride, rowb + (size_t)(base[b] + pth[d]) * row_stride, row_bytes);
    }
    return skipped;
}

/* ------------------------------------------------- draft sampling + verify */

/*
 * The draft side of a round done in the same call as the verify: each drafted token
 * x_k is drawn from q_k = softmax(draft_logits_k / T) ("[논문 리뷰] Fast Inference
 * from Transformers via Speculative Decoding", section 2, Step 1: the draft model
 * proposes x_1..x_K by sampling; "Speculative Decoding and EAGLE", section "개념"),
 * then the K tokens are verified exactly as oracle_verify_chain does with the
 * drafts given as logits.  The draft uniform of position k is word 2 of Philox slot
 * k (words 0 and 1 stay the accept and draw uniforms), on the same 24-bit grid; the
 * token is the inverse-CDF draw of that uniform from q_k.  Greedy rows (T <= 0)
 * draft x_k = argmax of draft row k (lowest index on ties) and verify greedily.
 *  target [B][K+1][V], draft [B][K][V] logits; out_draft_tokens [B][K] (-1 for a
 *  draft row that is invalid data, which makes the whole batch row invalid);
 *  other outputs as oracle_verify_chain.  out_margin also covers the draft draws.
 */
int oracle_sample_and_verify(const void *target, int tdt, const void *draft, int ddt,
                             const float *temperature, int B, int K, int V, uint64_t seed,
                             uint64_t offset, const int32_t *row_id, int32_t *out_draft_tokens,
                             int32_t *out_tokens, int32_t *out_count, float *out_accept_prob,
                             double *out_margin)
{
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    int n_invalid = 0;
    for (int b = 0; b < B; ++b) {
        const uint64_t rid = row_id ? (uint64_t)row_id[b] : (uint64_t)b;
        const double T = (double)temperature[b];
        const int greedy = !(T > 0.0);
        int32_t *xd = out_draft_tokens + (size_t)b * K;
        double margin = INFINITY;
        for (int k = 0; k < K; ++k) {
            const size_t off = ((size_t)b * K + k) * (size_t)V;
            if (greedy) {
                double m;
                int g;
                xd[k] = orc_row_max(draft, ddt, off, V, &m, &g) ? -1 : g;
                continue;
            }
            if (orc_softmax(draft, ddt, off, V, T, q)) { xd[k] = -1; continue; }
            uint64_t c[4] = {(uint64_t)k, rid, offset, 0}, key[2] = {seed, 0}, w[4];
            oracle_philox4x64_10(c, key, w);
            double mg;
            xd[k] = orc_draw(q, V, orc_u24(w[2]), &mg);
            margin = orc_min(margin, mg);
        }
        const size_t tro = (size_t)b * (K + 1) * (size_t)V, dro = (size_t)b * K * (size_t)V;
        const size_t tsz = tdt == ORC_F32 ? 4 : 2, dsz = ddt == ORC_F32 ? 4 : 2;
        double vm = INFINITY;
        const int32_t rid32 = (int32_t)rid;
        n_invalid += oracle_verify_chain((const char *)target + tro * tsz, tdt, (const char *)draft + dro * dsz,
                                         ddt, ORC_DRAFT_LOGITS, xd, temperature + b, 1, K, V, seed, offset,
                                         &rid32, out_tokens + (size_t)b * (K + 1), out_count + b,
                                         out_accept_prob ? out_accept_prob + (size_t)b * (K > 0 ? K : 1) : NULL,
                                         &vm);
        if (out_margin) out_margin[b] = orc_min(margin, vm);
    }
    free(q);
    return n_invalid;
}
