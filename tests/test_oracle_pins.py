"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties the oracle to a library routine, a closed form, an exact law
enumeration, a statistical law, or a brute-force search, chosen so that a
plausible slip (a wrong temperature, the scalar-q residual, an off-by-one
position, <= instead of <, a wrong Philox word) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth

GRID = 1 << 24  # uniforms live on the 24-bit grid n * 2^-24
HERE = os.path.dirname(os.path.abspath(__file__))


def softmax64(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


# ------------------------------------------------------------------ Philox

def test_philox_matches_numpy_philox():
    """Philox4x64-10 block == numpy.random.Philox (which returns the block of counter+1)."""
    rng = np.random.default_rng(1)
    cases = [([0, 0, 0, 0], [0, 0]), ([2**64 - 1] * 4, [2**64 - 1] * 2)]
    for _ in range(20):
        cases.append((list(rng.integers(0, 2**63, 4, dtype=np.uint64) * 2 + 1),
                      list(rng.integers(0, 2**63, 2, dtype=np.uint64))))
    cases.append(([5, 3, 9, 0], [12345, 0]))
    for ctr, key in cases:
        ctr = [int(c) for c in ctr]
        # numpy increments the 256-bit counter before producing a block: pass ctr - 1.
        val = ctr[0] + (ctr[1] << 64) + (ctr[2] << 128) + (ctr[3] << 192)
        val = (val - 1) % (1 << 256)
        prev = [(val >> (64 * i)) & (2**64 - 1) for i in range(4)]
        ref = np.random.Philox(counter=np.array(prev, np.uint64),
                              key=np.array([int(k) for k in key], np.uint64)).random_raw(4)
        got = oracle.philox4x64_10(ctr, key)
        assert [int(x) for x in got] == [int(x) for x in ref]


def test_accept_uniform_is_word0_slot_k():
    """Position k's accept uniform is (w0 >> 40) * 2^-24 of block {k, row, offset, 0}:
    driving the oracle with those uniforms explicitly gives the same outputs."""
    w = synth.tiny_chain(seed=3, V=16, K=3, B=5)
    seed, offset = 77, 4
    r = np.zeros((5, 3))
    u = np.zeros((5, 4))
    for b in range(5):
        for k in range(4):
            blk = oracle.philox4x64_10([k, b, offset, 0], [seed, 0])
            if k < 3:
                r[b, k] = int(blk[0] >> np.uint64(40)) / GRID
            u[b, k] = int(blk[1] >> np.uint64(40)) / GRID
    a = oracle.verify_chain(w["target"], w["draft"], w["tokens"], w["temperature"], seed, offset)
    e = oracle.verify_chain(w["target"], w["draft"], w["tokens"], w["temperature"], 0, 0, uniforms=(r, u))
    assert np.array_equal(a["tokens"], e["tokens"]) and np.array_equal(a["count"], e["count"])


# -------------------------------------------------------- softmax / ratio

@pytest.mark.parametrize("T", [0.25, 0.8, 1.0, 1.5, 3.0])
def test_acceptance_probability_is_logistic_for_two_tokens(T):
    """V=2, q = (1, 0), x = 0: the acceptance probability is p(0) = 1/(1+exp((b-a)/T))."""
    rng = np.random.default_rng(int(T * 100))
    B = 64
    ab = rng.normal(0, 3, (B, 2)).astype(np.float32)
    target = np.repeat(ab[:, None, :], 2, axis=1)  # K = 1
    draft = np.tile(np.array([1.0, 0.0], np.float32), (B, 1, 1))
    toks = np.zeros((B, 1), np.int32)
    out = oracle.verify_chain(target, draft, toks, np.full(B, T, np.float32), 1, 0,
                              draft_kind=oracle.DRAFT_PROBS)
    expect = 1.0 / (1.0 + np.exp((ab[:, 1].astype(np.float64) - ab[:, 0]) / np.float32(T)))
    np.testing.assert_allclose(out["accept_prob"][:, 0], expect, rtol=0, atol=1e-7)


def test_shift_invariance_and_constant_rows():
    """Adding a constant to every logit of a row changes nothing; constant logits give
    p = 1/V, so with q = p every draft is accepted."""
    w = synth.tiny_chain(seed=5, V=32, K=3, B=40)
    base = oracle.verify_chain(w["target"], w["draft"], w["tokens"], w["temperature"], 9, 1)
    shifted = oracle.verify_chain(w["target"] + np.float32(8.0), w["draft"] - np.float32(4.0),
                                  w["tokens"], w["temperature"], 9, 1)
    assert np.array_equal(base["tokens"], shifted["tokens"])
    V, K, B = 16, 3, 10
    target = np.zeros((B, K + 1, V), np.float32)
    draft = np.full((B, K, V), 1.0 / V, np.float32)
    toks = np.random.default_rng(0).integers(0, V, (B, K)).astype(np.int32)
    out = oracle.verify_chain(target, draft, toks, np.ones(B, np.float32), 3, 0,
                              draft_kind=oracle.DRAFT_PROBS)
    assert (out["count"] == K + 1).all()
    np.testing.assert_array_equal(out["accept_prob"], np.ones((B, K), np.float32))


def test_strict_less_than_at_the_boundary():
    """Logits (0, 0) give p = (1/2, 1/2); q = (1, 0) gives ratio 1/2 exactly:
    r = 1/2 rejects (accept iff r < ratio), the grid point below accepts."""
    target = np.zeros((2, 2, 2), np.float32)
    draft = np.tile(np.array([1.0, 0.0], np.float32), (2, 1, 1))
    toks = np.zeros((2, 1), np.int32)
    r = np.array([[0.5], [0.5 - 1.0 / GRID]])
    u = np.full((2, 2), 0.25)
    out = oracle.verify_chain(target, draft, toks, np.ones(2, np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(r, u))
    assert out["count"].tolist() == [1, 2]
    assert out["tokens"][0, 0] == 1  # residual (p - q)+ = (0, 1/2): only token 1
    assert out["tokens"][1, 0] == 0


# ------------------------------------------------------------- the draw

def test_residual_draw_matches_searchsorted():
    """The replacement is searchsorted(cumsum(max(0, p - q)), u * Z, 'right') with p a known
    distribution (logits = log w) and q given -- the full q vector, not q(x) alone."""
    rng = np.random.default_rng(11)
    V, B = 12, 300
    wts = rng.gamma(0.7, size=(B, V)) + 1e-3
    p = wts / wts.sum(1, keepdims=True)
    q = rng.dirichlet(np.ones(V) * 0.5, size=B)
    target = np.zeros((B, 2, V), np.float32)
    target[:, 0] = np.log(wts).astype(np.float32)
    p = np.stack([softmax64(np.log(wts[b]).astype(np.float32)) for b in range(B)])
    x = np.array([int(np.argmax(q[b] - p[b])) for b in range(B)], np.int32)  # ratio < 1
    r = np.full((B, 1), 1.0 - 1.0 / GRID)  # force rejection
    u = np.stack([rng.integers(0, GRID, B) / GRID, np.zeros(B)], 1)
    out = oracle.verify_chain(target, q[:, None, :].astype(np.float32), x[:, None],
                              np.ones(B, np.float32), 0, 0, draft_kind=oracle.DRAFT_PROBS,
                              uniforms=(r, u))
    q32 = q.astype(np.float32).astype(np.float64)
    for b in range(B):
        res = np.maximum(p[b] - q32[b], 0.0)
        expect = int(np.searchsorted(np.cumsum(res), u[b, 0] * res.sum(), side="right"))
        assert out["count"][b] == 1
        assert out["tokens"][b, 0] == expect


def test_bonus_draw_matches_searchsorted():
    """p == q accepts every draft (ratio exactly 1); the bonus token is the inverse-CDF draw
    from p at position K."""
    rng = np.random.default_rng(12)
    B, K, V = 200, 3, 20
    target = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    draft = target[:, :K].copy()
    toks = rng.integers(0, V, (B, K)).astype(np.int32)
    T = np.float32(0.7)
    u = rng.integers(0, GRID, (B, K + 1)) / GRID
    r = rng.integers(0, GRID, (B, K)) / GRID
    out = oracle.verify_chain(target, draft, toks, np.full(B, T, np.float32), 0, 0, uniforms=(r, u))
    assert (out["count"] == K + 1).all()
    for b in range(B):
        assert out["tokens"][b, :K].tolist() == toks[b].tolist()
        pK = softmax64(target[b, K].astype(np.float64) / np.float64(T))
        expect = int(np.searchsorted(np.cumsum(pK), u[b, K] * pK.sum(), side="right"))
        assert out["tokens"][b, K] == expect


def test_disjoint_supports_give_one_token_from_p():
    """q and p on disjoint supports: every draft is rejected, the replacement (the residual
    is p itself) always lies in p's support, and it is distributed as p_0.  Every row
    shares one target row 0, so the B replacements are B draws from one law, checked by a
    chi-square test over the half support (7 degrees of freedom; 24.32 is the 0.999
    quantile of that law)."""
    rng = np.random.default_rng(13)
    B, K, V = 4000, 4, 16
    target = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    target[:, 0] = rng.normal(0, 1, V).astype(np.float32)  # one row 0 for every batch row
    draft = rng.normal(0, 1, (B, K, V)).astype(np.float32)
    target[:, :, V // 2:] = -np.inf
    draft[:, :, : V // 2] = -np.inf
    toks = rng.integers(V // 2, V, (B, K)).astype(np.int32)
    out = oracle.verify_chain(target, draft, toks, np.ones(B, np.float32), 21, 0)
    assert (out["count"] == 1).all()
    assert (out["tokens"][:, 0] < V // 2).all() and (out["tokens"][:, 0] >= 0).all()
    # law of the replacement is p_0: chi-square over the half support
    counts = np.bincount(out["tokens"][:, 0], minlength=V)[: V // 2]
    p0 = softmax64(target[0, 0, : V // 2].astype(np.float64))
    expected = B * p0
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 24.32, (chi2, counts.tolist(), expected.round(1).tolist())
    # the same statistic rejects a plausible slip: a replacement drawn uniformly over the support
    uniform = np.full(V // 2, B / (V // 2))
    assert float(((counts - uniform) ** 2 / uniform).sum()) > 24.32


# ------------------------------------------- exact law on the uniform grid

def _bisect_first_true(pred_batch, n_rows):
    """For monotone predicates f_j(n) on n in [0, GRID] (False ... False True ... True),
    return for every j the smallest n with f_j(n) True (GRID if none)."""
    lo = np.full(n_rows, -1, np.int64)
    hi = np.full(n_rows, GRID, np.int64)
    while (hi - lo > 1).any():
        mid = (lo + hi) // 2
        active = hi - lo > 1
        res = pred_batch(np.where(active, mid, 0))
        hi = np.where(active & res, mid, hi)
        lo = np.where(active & ~res, mid, lo)
    return hi


def _chain_law_k1(target_row0, target_row1, qrow, draft_logits_row, T, dk):
    """Black-box exact law of the first emitted token and of the bonus token for K=1, by
    bisection of the oracle's outcome over the 24-bit grids of r and u."""
    V = target_row0.size
    q = qrow
    xs = [x for x in range(V) if q[x] > 0]
    target = np.stack([target_row0, target_row1])[None]
    drow = (draft_logits_row if dk == oracle.DRAFT_LOGITS else q.astype(np.float32))[None, None]

    def run(rr, uu, x):
        n = len(rr)
        return oracle.verify_chain(np.repeat(target, n, 0), np.repeat(drow, n, 0),
                                   np.asarray(x, np.int32)[:, None], np.full(n, T, np.float32), 0, 0,
                                   draft_kind=dk, uniforms=(np.asarray(rr)[:, None],
                                                            np.stack([uu, uu], 1)))

    X = np.array(xs)
    # P(accept | x): smallest grid r that rejects
    first_reject = _bisect_first_true(lambda n: run(n / GRID, np.zeros(len(X)), X)["count"] == 1, len(X))
    p_acc = first_reject / GRID
    # replacement law | x: breakpoints of the (monotone) drawn token in u
    pairs = [(x, i) for x in xs for i in range(1, V)]
    PX = np.array([a for a, _ in pairs])
    PI = np.array([b for _, b in pairs])
    rej_r = np.full(len(pairs), 1.0 - 1.0 / GRID)
    bp = _bisect_first_true(lambda n: run(rej_r, n / GRID, PX)["tokens"][:, 0] >= PI, len(pairs))
    law = np.zeros(V)
    for j, x in enumerate(xs):
        law[x] += q[x] * p_acc[j]
        if p_acc[j] < 1.0:
            b = np.concatenate([[0], bp[j * (V - 1):(j + 1) * (V - 1)], [GRID]])
            law += q[x] * (1 - p_acc[j]) * np.diff(b) / GRID
    # bonus law: force acceptance (r = 0) of a token with p > 0
    xacc = np.full(V - 1, xs[int(np.argmax(p_acc))])
    bb = _bisect_first_true(lambda n: run(np.zeros(V - 1), n / GRID, xacc)["tokens"][:, 1] >= np.arange(1, V),
                            V - 1)
    bonus = np.diff(np.concatenate([[0], bb, [GRID]])) / GRID
    return law, bonus


@pytest.mark.parametrize("V,T,dk", [(8, 1.0, oracle.DRAFT_LOGITS), (6, 0.7, oracle.DRAFT_LOGITS),
                                    (8, 1.3, oracle.DRAFT_PROBS), (5, 1.0, oracle.DRAFT_PROBS)])
def test_exact_output_law_equals_p(V, T, dk):
    """Losslessness: enumerating the oracle over the uniform grid, the first emitted token has
    law p_0 and the bonus token law p_1 (up to the 2^-24 grid)."""
    rng = np.random.default_rng(V * 10 + int(T * 10))
    t0 = rng.normal(0, 2, V).astype(np.float32)
    t1 = rng.normal(0, 2, V).astype(np.float32)
    dl = (t0 + rng.normal(0, 1.0, V)).astype(np.float32)
    if dk == oracle.DRAFT_LOGITS:
        q = softmax64(dl.astype(np.float64) / np.float64(np.float32(T)))
    else:
        q = rng.dirichlet(np.ones(V)).astype(np.float32).astype(np.float64)
        q[0] = 0.0  # a zero-probability draft token is never drafted
        q = (q / q.sum()).astype(np.float32).astype(np.float64)
    law, bonus = _chain_law_k1(t0, t1, q, dl, np.float32(T), dk)
    p0 = softmax64(t0.astype(np.float64) / np.float64(np.float32(T)))
    p1 = softmax64(t1.astype(np.float64) / np.float64(np.float32(T)))
    np.testing.assert_allclose(law, p0, atol=4e-6)
    np.testing.assert_allclose(bonus, p1, atol=4e-6)


# ------------------------------------------------ expected tokens per round

def _golden_expected():
    rows = []
    with open(os.path.join(HERE, "golden", "expected_tokens.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, k, e, tol = line.split()
                rows.append((float(a), int(k), float(e), float(tol)))
    return rows


def _two_token_chain(alpha, K, n_rounds):
    """p = (alpha, 1 - alpha), q = (1, 0), x = 0 at every position: acceptance prob alpha."""
    target = np.tile(np.log(np.array([alpha, 1 - alpha], np.float64)).astype(np.float32), (n_rounds, K + 1, 1))
    draft = np.tile(np.array([1.0, 0.0], np.float32), (n_rounds, K, 1))
    return target, draft, np.zeros((n_rounds, K), np.int32)


def test_expected_tokens_matches_pages_worked_example():
    for alpha, K, printed, tol in _golden_expected():
        assert abs((1 - alpha ** (K + 1)) / (1 - alpha) - printed) <= tol
        n = 20000
        target, draft, toks = _two_token_chain(alpha, K, n)
        out = oracle.verify_chain(target, draft, toks, np.ones(n, np.float32), 2024, 0,
                                  draft_kind=oracle.DRAFT_PROBS)
        c = out["count"].astype(np.float64)
        se = c.std() / math.sqrt(n)
        assert abs(c.mean() - printed) < 4 * se + tol


@pytest.mark.parametrize("alpha", [0.5, 0.7, 0.9])
@pytest.mark.parametrize("K", [1, 3, 5, 8])
def test_expected_tokens_closed_form(alpha, K):
    n = 10000
    target, draft, toks = _two_token_chain(alpha, K, n)
    out = oracle.verify_chain(target, draft, toks, np.ones(n, np.float32), 7 + K, 3,
                              draft_kind=oracle.DRAFT_PROBS)
    c = out["count"].astype(np.float64)
    expect = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(c.mean() - expect) < 4 * c.std() / math.sqrt(n) + 1e-9
    # the count law itself is a truncated geometric
    for j in range(1, K + 2):
        pj = alpha ** (j - 1) * ((1 - alpha) if j <= K else 1.0)
        emp = (out["count"] == j).mean()
        assert abs(emp - pj) < 4 * math.sqrt(pj * (1 - pj) / n) + 1e-9


def _fixed_rows_fresh_drafts(V, K, n, seed, T=1.0, sigma=0.5):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    d = (t[:K] + rng.normal(0, sigma, (K, V))).astype(np.float32)
    toks = np.stack([synth.draft_tokens_from_logits(rng, d, T) for _ in range(n)])
    return np.broadcast_to(t, (n, K + 1, V)).copy(), np.broadcast_to(d, (n, K, V)).copy(), toks


def test_expected_tokens_with_per_position_alpha():
    """E[count] = sum_j prod_{i<j} alpha_i with alpha_i = sum_x min(p_i(x), q_i(x))."""
    V, K, n = 8, 4, 20000
    target, draft, toks = _fixed_rows_fresh_drafts(V, K, n, seed=31)
    out = oracle.verify_chain(target, draft, toks, np.ones(n, np.float32), 99, 0)
    alphas = [np.minimum(softmax64(target[0, i]), softmax64(draft[0, i])).sum() for i in range(K)]
    expect = sum(np.prod(alphas[:j]) for j in range(K + 1))
    c = out["count"].astype(np.float64)
    assert abs(c.mean() - expect) < 4 * c.std() / math.sqrt(n)


def test_mean_accept_prob_at_a_position_estimates_its_alpha():
    """With x_k drawn from q_k, the mean of the reported min(1, p_k(x_k)/q_k(x_k)) is
    alpha_k = sum_x min(p_k(x), q_k(x)) (sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p, q)).
    Position 0 is evaluated in every round; at later positions only rounds that reached
    them report a value, and x_k is drawn independently of earlier decisions, so the
    conditional mean has the same expectation."""
    V, K, n = 8, 3, 20000
    target, draft, toks = _fixed_rows_fresh_drafts(V, K, n, seed=37, sigma=1.0)
    out = oracle.verify_chain(target, draft, toks, np.ones(n, np.float32), 5, 0)
    ap = out["accept_prob"].astype(np.float64)
    for k in range(K):
        alpha = np.minimum(softmax64(target[0, k]), softmax64(draft[0, k])).sum()
        got = ap[ap[:, k] >= 0, k]
        assert len(got) > 1000
        assert abs(got.mean() - alpha) < 4 * got.std() / math.sqrt(len(got)), (k, got.mean(), alpha)


# ---------------------------------------------------------- distribution

def test_tv_distance_first_and_second_token():
    """Exercise 1 of the EAGLE lesson: the emitted tokens follow the target law.  TV of the
    first token against p_0 is within the 99th percentile of an exact sampler's TV at the same
    n; the second token (after an accepted first draft) follows p_1; chi-square passes."""
    scipy_stats = pytest.importorskip("scipy.stats")
    V, K = 8, 4
    rng = np.random.default_rng(5)
    for n in (10_000, 400_000):
        target, draft, toks = _fixed_rows_fresh_drafts(V, K, n, seed=41)
        out = oracle.verify_chain(target, draft, toks, np.ones(n, np.float32), 1234, n)
        p0 = softmax64(target[0, 0])
        emp = np.bincount(out["tokens"][:, 0], minlength=V) / n
        tv = 0.5 * np.abs(emp - p0).sum()
        exact_tv = [0.5 * np.abs(rng.multinomial(n, p0) / n - p0).sum() for _ in range(400)]
        assert tv <= np.quantile(exact_tv, 0.99)
        if n >= 100_000:
            assert tv < 0.01
        chi = scipy_stats.chisquare(np.bincount(out["tokens"][:, 0], minlength=V), p0 * n)
        assert chi.pvalue > 1e-3
        sel = out["count"] >= 2
        p1 = softmax64(target[0, 1])
        m = int(sel.sum())
        emp1 = np.bincount(out["tokens"][sel, 1], minlength=V) / m
        exact_tv1 = [0.5 * np.abs(rng.multinomial(m, p1) / m - p1).sum() for _ in range(400)]
        assert 0.5 * np.abs(emp1 - p1).sum() <= np.quantile(exact_tv1, 0.995)


# ---------------------------------------------------------------- greedy

def test_greedy_matches_numpy_argmax_with_ties():
    rng = np.random.default_rng(8)
    B, K, V = 300, 5, 24
    vals = rng.integers(-3, 3, (B, K + 1, V)).astype(np.float32)  # many ties
    target = synth.f32_to_bf16_bits(vals)
    am = np.argmax(vals, axis=2)
    toks = am[:, :K].copy()
    cut = rng.integers(0, K + 1, B)
    for b in range(B):
        if cut[b] < K:
            toks[b, cut[b]] = (am[b, cut[b]] + 1 + rng.integers(0, V - 1)) % V
    out = oracle.greedy_accept(target, toks.astype(np.int32))
    for b in range(B):
        j = int(cut[b])
        assert out["count"][b] == j + 1
        assert out["tokens"][b, :j].tolist() == am[b, :j].tolist()
        assert out["tokens"][b, j] == am[b, j]
        assert (out["tokens"][b, j + 1:] == -1).all()
    # temperature 0 rows of verify_chain follow the same rule and never read the draft
    ch = oracle.verify_chain(target, None, toks.astype(np.int32), np.zeros(B, np.float32), 0, 0)
    assert np.array_equal(ch["tokens"], out["tokens"]) and np.array_equal(ch["count"], out["count"])


# ----------------------------------------------------------------- trees

def _random_tree(rng, N, V):
    """Random parent array (parent[i] < i) with distinct sibling tokens."""
    parent = np.empty(N, np.int32)
    tokens = np.empty(N, np.int32)
    for i in range(N):
        open_nodes = [a for a in range(-1, i) if sum(parent[j] == a for j in range(i)) < V]
        parent[i] = open_nodes[rng.integers(0, len(open_nodes))]
        used = {int(tokens[j]) for j in range(i) if parent[j] == parent[i]}
        tokens[i] = rng.choice([v for v in range(V) if v not in used])
    return tokens, parent


def test_greedy_tree_is_longest_matching_branch_brute_force():
    rng = np.random.default_rng(17)
    B, N, V = 200, 12, 4
    target = rng.integers(0, 3, (B, N + 1, V)).astype(np.float32)
    toks = np.empty((B, N), np.int32)
    par = np.empty((B, N), np.int32)
    for b in range(B):
        toks[b], par[b] = _random_tree(rng, N, V)
    depth = np.zeros((B, N), int)
    for b in range(B):
        for i in range(N):
            depth[b, i] = 1 if par[b, i] < 0 else depth[b, par[b, i]] + 1
    D = int(depth.max())
    out = oracle.verify_tree(target, None, toks, par, np.zeros(B, np.float32), D, 0, 0)
    for b in range(B):
        am = np.argmax(target[b], axis=1)  # am[row]; row of node i is i + 1, root row 0
        best = []
        for i in range(N):  # enumerate every root path, keep those whose nodes all match
            path, node = [], i
            while node >= 0:
                path.append(node)
                node = par[b, node]
            path = path[::-1]
            ok = all(toks[b, a] == am[0 if par[b, a] < 0 else par[b, a] + 1] for a in path)
            if ok and len(path) > len(best):
                best = path
        end_row = 0 if not best else best[-1] + 1
        expect = [int(toks[b, a]) for a in best] + [int(am[end_row])]
        assert out["count"][b] == len(expect)
        assert out["tokens"][b, : len(expect)].tolist() == expect
        assert out["path"][b, : len(best)].tolist() == best


@pytest.mark.parametrize("T,kind", [(1.0, "logits"), (0.7, "probs"), (0.0, "logits")])
def test_chain_as_tree_reproduces_chain(T, kind):
    if kind == "logits":
        w = synth.tiny_chain(seed=23, V=64, K=4, B=300, temperature=T)
    else:
        w = synth.single_stream(seed=23, V=64, K=4, B=300, temperature=T)
    tw = synth.chain_as_tree(w)
    c = oracle.verify_chain(w["target"], w["draft"], w["tokens"], w["temperature"], 5, 6,
                            draft_kind=w["draft_kind"])
    t = oracle.verify_tree(tw["target"], tw["draft"], tw["node_tokens"], tw["parent"], tw["temperature"],
                           tw["max_depth"], 5, 6, draft_kind=tw["draft_kind"])
    assert np.array_equal(c["tokens"], t["tokens"]) and np.array_equal(c["count"], t["count"])
    np.testing.assert_array_equal(c["margin"], t["margin"])


@pytest.mark.parametrize("V,T", [(5, 1.0), (4, 0.8)])
def test_tree_siblings_without_replacement_are_exact(V, T):
    """Root with two children drawn without replacement from q: enumerating the oracle over the
    uniform grids and over the ordered child pairs, the first emitted token has law p_root."""
    rng = np.random.default_rng(V + 100)
    t0 = rng.normal(0, 1.5, V).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 2).astype(np.float32).astype(np.float64)
    q = q / q.sum()
    q32 = q.astype(np.float32)
    pairs = [(a, c) for a in range(V) for c in range(V) if a != c]
    weight = np.array([q32[a] / q32.sum() * q32[c] / (q32.sum() - q32[a]) for a, c in pairs], np.float64)
    n = len(pairs)
    target = np.tile(np.stack([t0, t0, t0])[None], (n, 1, 1))
    draft = np.tile(np.stack([q32, q32, q32])[None], (n, 1, 1))
    toks = np.array(pairs, np.int32)
    par = np.full((n, 2), -1, np.int32)

    def run(r1, r2, u0):
        m = len(r1)
        idx = np.arange(m) % n
        return oracle.verify_tree(target[idx], draft[idx], toks[idx], par[idx], np.full(m, T, np.float32), 1,
                                  0, 0, draft_kind=oracle.DRAFT_PROBS,
                                  uniforms=(np.stack([r1, r2], 1), np.stack([u0, u0, u0], 1)))

    top = 1.0 - 1.0 / GRID
    first = _bisect_first_true(lambda k: run(k / GRID, np.zeros(n), np.zeros(n))["path"][:, 0] != 0, n)
    p1 = first / GRID
    second = _bisect_first_true(lambda k: run(np.full(n, top), k / GRID, np.zeros(n))["path"][:, 0] != 1, n)
    p2 = second / GRID
    rows = np.repeat(np.arange(n), V - 1)
    thr = np.tile(np.arange(1, V), n)

    def draw_pred(k):
        m = len(rows)
        out = oracle.verify_tree(target[rows], draft[rows], toks[rows], par[rows], np.full(m, T, np.float32), 1,
                                 0, 0, draft_kind=oracle.DRAFT_PROBS,
                                 uniforms=(np.full((m, 2), top), np.stack([k / GRID] * 3, 1)))
        return out["tokens"][:, 0] >= thr

    bp = _bisect_first_true(draw_pred, len(rows)).reshape(n, V - 1)
    law = np.zeros(V)
    for j, (a, c) in enumerate(pairs):
        res = np.diff(np.concatenate([[0], bp[j], [GRID]])) / GRID
        law[a] += weight[j] * p1[j]
        law[c] += weight[j] * (1 - p1[j]) * p2[j]
        law += weight[j] * (1 - p1[j]) * (1 - p2[j]) * res
    p = softmax64(t0.astype(np.float64) / np.float64(np.float32(T)))
    np.testing.assert_allclose(law, p, atol=5e-6)


def _root_two_children_law(t0, q32, T, pairs, weight, rule):
    """Exact law of the first emitted token of a root with two children whose token
    pairs come with the given weights, enumerating the oracle over the uniform grids."""
    V = t0.size
    n = len(pairs)
    target = np.tile(np.stack([t0, t0, t0])[None], (n, 1, 1))
    draft = np.tile(np.stack([q32, q32, q32])[None], (n, 1, 1))
    toks = np.array(pairs, np.int32)
    par = np.full((n, 2), -1, np.int32)

    def run(idx, r1, r2, u0):
        m = len(idx)
        return oracle.verify_tree(target[idx], draft[idx], toks[idx], par[idx], np.full(m, T, np.float32), 1,
                                  0, 0, draft_kind=oracle.DRAFT_PROBS, sibling_rule=rule,
                                  uniforms=(np.stack([r1, r2], 1), np.stack([u0, u0, u0], 1)))

    top = 1.0 - 1.0 / GRID
    idx = np.arange(n)
    p1 = _bisect_first_true(lambda k: run(idx, k / GRID, np.zeros(n), np.zeros(n))["path"][:, 0] != 0, n) / GRID
    p2 = _bisect_first_true(lambda k: run(idx, np.full(n, top), k / GRID, np.zeros(n))["path"][:, 0] != 1,
                            n) / GRID
    rows = np.repeat(idx, V - 1)
    thr = np.tile(np.arange(1, V), n)
    m = len(rows)
    bp = _bisect_first_true(lambda k: run(rows, np.full(m, top), np.full(m, top), k / GRID)["tokens"][:, 0] >= thr,
                            m).reshape(n, V - 1)
    law = np.zeros(V)
    for j, (a, c) in enumerate(pairs):
        res = np.diff(np.concatenate([[0], bp[j], [GRID]])) / GRID
        law[a] += weight[j] * p1[j]
        law[c] += weight[j] * (1 - p1[j]) * p2[j]
        law += weight[j] * (1 - p1[j]) * (1 - p2[j]) * res
    return law


@pytest.mark.parametrize("V,T", [(5, 1.0), (4, 0.8)])
def test_tree_siblings_iid_rule_is_exact_and_the_rules_differ(V, T):
    """Multi-draft verification with children drawn i.i.d. from q (repeats allowed): the
    i.i.d. rule (q left as it is after a rejection) gives law p_root exactly; the
    without-replacement rule applied to the same drafts does not, and neither does the
    i.i.d. rule applied to children drawn without replacement."""
    rng = np.random.default_rng(V + 200)
    t0 = rng.normal(0, 0.7, V).astype(np.float32)  # a flat p: the residual keeps several tokens
    q32 = (rng.dirichlet(np.ones(V) * 2)).astype(np.float32)
    q = q32.astype(np.float64) / q32.astype(np.float64).sum()
    p = softmax64(t0.astype(np.float64) / np.float64(np.float32(T)))
    iid_pairs = [(a, c) for a in range(V) for c in range(V)]
    iid_w = np.array([q[a] * q[c] for a, c in iid_pairs])
    law_iid = _root_two_children_law(t0, q32, T, iid_pairs, iid_w, oracle.SIBLINGS_IID)
    np.testing.assert_allclose(law_iid, p, atol=5e-6)
    law_mixed = _root_two_children_law(t0, q32, T, iid_pairs, iid_w, oracle.SIBLINGS_WOR)
    assert np.abs(law_mixed - p).max() > 1e-3
    wor_pairs = [(a, c) for a in range(V) for c in range(V) if a != c]
    wor_w = np.array([q[a] * q[c] / (1 - q[a]) for a, c in wor_pairs])
    law_wor = _root_two_children_law(t0, q32, T, wor_pairs, wor_w, oracle.SIBLINGS_WOR)
    np.testing.assert_allclose(law_wor, p, atol=5e-6)
    assert np.abs(_root_two_children_law(t0, q32, T, wor_pairs, wor_w, oracle.SIBLINGS_IID) - p).max() > 1e-3


def test_sibling_rules_agree_for_a_single_child_and_on_chains():
    """The two rules differ only after a rejection among siblings: with at most one
    child per node (a chain) they give identical results."""
    w = synth.chain_as_tree(synth.tiny_chain(seed=8, V=64, K=4, B=40))
    args = (w["target"], w["draft"], w["node_tokens"], w["parent"], w["temperature"], w["max_depth"], 3, 1)
    a = oracle.verify_tree(*args, draft_kind=w["draft_kind"], sibling_rule=oracle.SIBLINGS_WOR)
    b = oracle.verify_tree(*args, draft_kind=w["draft_kind"], sibling_rule=oracle.SIBLINGS_IID)
    for k in ("tokens", "count", "path", "margin"):
        np.testing.assert_array_equal(a[k], b[k])


# ------------------------------------------------------------ bad inputs

def test_invalid_rows_give_count_zero():
    w = synth.tiny_chain(seed=2, V=16, K=3, B=6)
    t = w["target"].copy()
    toks = w["tokens"].copy()
    t[0, 0, 3] = np.nan          # NaN in the first row read
    t[1, 0, :] = -np.inf         # all -inf
    t[2, 0, 5] = np.inf          # +inf
    toks[3, 2] = 16              # token out of range
    t[4, 3, :] = np.nan          # a row that is never reached when the round stops earlier
    out = oracle.verify_chain(t, w["draft"], toks, w["temperature"], 1, 0)
    assert out["count"][:4].tolist() == [0, 0, 0, 0]
    assert (out["tokens"][:4] == -1).all()
    assert out["n_invalid"] >= 4
    assert out["count"][5] >= 1
    # masked (-inf) entries are fine and never drawn
    t2 = w["target"].copy()
    t2[:, :, :8] = -np.inf
    out2 = oracle.verify_chain(t2, w["draft"], w["tokens"], w["temperature"], 1, 0)
    assert (out2["count"] >= 1).all()
    for b in range(6):
        c = out2["count"][b]
        assert out2["tokens"][b, c - 1] >= 8


def test_malformed_tree_is_invalid():
    rng = np.random.default_rng(3)
    V, N = 10, 5
    target = rng.normal(0, 1, (3, N + 1, V)).astype(np.float32)
    toks = np.tile(np.arange(N, dtype=np.int32), (3, 1))
    par = np.array([[-1, 0, 1, 2, 3], [-1, 0, 2, 1, 0], [-1, 0, 1, 2, 3]], np.int32)  # row 1: parent[2]=2
    out = oracle.verify_tree(target, None, toks, par, np.zeros(3, np.float32), 5, 0, 0)
    assert out["count"][1] == 0 and out["count"][0] >= 1
    out = oracle.verify_tree(target, None, toks, par, np.zeros(3, np.float32), 3, 0, 0)  # depth 5 > 3
    assert out["count"][0] == 0


def test_margin_reports_distance_to_decision():
    """margin = |r - ratio| for an accept decision; the CDF distance for a draw."""
    target = np.zeros((1, 2, 2), np.float32)
    draft = np.array([[[1.0, 0.0]]], np.float32)
    r = np.array([[0.375]])
    u = np.array([[0.0, 0.25]])
    out = oracle.verify_chain(target, draft, np.zeros((1, 1), np.int32), np.ones(1, np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(r, u))
    # ratio 0.5 accepted with margin 0.125; bonus draw from (1/2, 1/2) at t = 0.25 -> margin 0.25
    assert out["count"][0] == 2
    assert out["margin"][0] == pytest.approx(0.125, abs=1e-15)


def test_draw_margin_is_the_distance_to_the_nearest_cdf_boundary_in_mass():
    """Where the draw decides the margin: a bonus draw from p = (1/4)x4 at u = 0.26 lands
    0.01 past the boundary 0.25; a residual draw from (p - q)+ = (0, 1/2) at u = 0.9
    lands at t = u Z = 0.45, 0.05 (in mass, not divided by Z) below the boundary 0.5."""
    out = oracle.verify_chain(np.zeros((1, 1, 4), np.float32), np.zeros((1, 0, 4), np.float32),
                              np.zeros((1, 0), np.int32), np.ones(1, np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(np.zeros((1, 0)), np.array([[0.26]])))
    assert out["count"][0] == 1 and out["tokens"][0, 0] == 1
    assert out["margin"][0] == pytest.approx(0.01, abs=1e-12)
    out = oracle.verify_chain(np.zeros((1, 2, 2), np.float32), np.array([[[1.0, 0.0]]], np.float32),
                              np.zeros((1, 1), np.int32), np.ones(1, np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(np.array([[0.75]]), np.array([[0.9, 0.0]])))
    assert out["count"][0] == 1 and out["tokens"][0, 0] == 1  # x = 0 rejected (ratio 1/2), residual draws 1
    assert out["margin"][0] == pytest.approx(0.05, abs=1e-12)  # min(|0.75 - 0.5|, 0.05)


def test_accept_prob_layout_after_the_first_rejection_and_on_greedy_rows():
    """Sampling rows: min(1, p/q) up to and including the first rejection, -1 after it.
    Greedy rows: 1 for each match, 0 for the mismatch, -1 after it."""
    V, K = 3, 3
    target = np.zeros((2, K + 1, V), np.float32)
    target[1, :, 2] = 5.0  # greedy row: argmax 2 at every position
    draft = np.full((2, K, V), 1.0 / 3, np.float32)
    toks = np.array([[0, 1, 2], [2, 0, 2]], np.int32)
    r = np.array([[0.5, 0.9999, 0.0], [0.0, 0.0, 0.0]])  # row 0: ratio 1 at every position
    u = np.zeros((2, K + 1))
    out = oracle.verify_chain(target, draft, toks, np.array([1.0, 0.0], np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(r, u))
    # row 0: p = q = 1/3, ratio 1 > r: all accepted, then the bonus token
    assert out["count"][0] == K + 1
    np.testing.assert_array_equal(out["accept_prob"][0], [1.0, 1.0, 1.0])
    # row 1 (greedy): x_0 = 2 matches, x_1 = 0 does not -> emits 2; position 2 never evaluated
    assert out["count"][1] == 2 and list(out["tokens"][1, :2]) == [2, 2]
    np.testing.assert_array_equal(out["accept_prob"][1], [1.0, 0.0, -1.0])
    # a sampling row rejected at position 1 reports min(1, p/q) there and -1 after it
    target2 = np.zeros((1, K + 1, V), np.float32)
    target2[0, 1, 0] = -np.inf  # p_1(0) = 0, so x_1 = 0 is rejected (ratio 0)
    out = oracle.verify_chain(target2, draft[:1], np.array([[1, 0, 1]], np.int32), np.ones(1, np.float32), 0, 0,
                              draft_kind=oracle.DRAFT_PROBS, uniforms=(np.array([[0.3, 0.3, 0.3]]), np.zeros((1, K + 1))))
    assert out["count"][0] == 2
    np.testing.assert_array_equal(out["accept_prob"][0], [1.0, 0.0, -1.0])


def test_tree_margin_and_sibling_update_worked_example():
    """Root p = (1/2, 1/2), q = (3/4, 1/4); children x = 0 then x = 1.  Child 0: ratio 2/3,
    r = 0.9 rejects (margin 0.2333).  Then p <- (p - q)+ / Z = (0, 1), q(0) <- 0 and
    q <- q / sum q = (0, 1), so child 1 has ratio 1 and r = 0.4 accepts (margin 0.6).  Child
    1 is a leaf: the last token is drawn from its row p = (1/2, 1/2) at u = 0.7 -> token 1,
    margin 0.2.  The row's margin is the smallest, 0.2."""
    target = np.zeros((1, 3, 2), np.float32)
    draft = np.array([[[0.75, 0.25], [0.5, 0.5], [0.5, 0.5]]], np.float32)
    out = oracle.verify_tree(target, draft, np.array([[0, 1]], np.int32), np.array([[-1, -1]], np.int32),
                             np.ones(1, np.float32), 1, 0, 0, draft_kind=oracle.DRAFT_PROBS,
                             uniforms=(np.array([[0.9, 0.4]]), np.array([[0.0, 0.0, 0.7]])))
    assert out["count"][0] == 2
    assert list(out["tokens"][0]) == [1, 1] and list(out["path"][0]) == [1]
    assert out["margin"][0] == pytest.approx(0.2, abs=1e-12)
