"""Property checks of the oracle over random small cases (no GPU; skipped where the
hypothesis package is missing).

Each property follows from the rule alone, so it pins the oracle independently of
its own arithmetic:
- outputs are well formed (count in 1..K+1, kept drafts first, -1 padding);
- a chain given as a tree (parent[i] = i - 1) gives the same result bit for bit,
  the slot layout making the two walks consume the same uniforms;
- identical draft and target distributions accept every draft (ratio 1 > r);
- drafts outside the target's support are rejected at once, and the replacement lies
  in the support;
- the tree mask of any valid parent array is each node's ancestor-or-self set;
- the compaction of any root-to-node path is a gather from the unmodified cache.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


def _chain(seed, B, K, V, T, mask_frac):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    if mask_frac > 0:
        m = rng.random((B, K + 1, V)) < mask_frac
        m[..., 0] = False  # keep one finite logit per row
        t[m] = -np.inf
    toks = rng.integers(0, V, (B, K)).astype(np.int32)
    temps = np.full(B, T, np.float32)
    return t, d, toks, temps


cases = st.tuples(st.integers(0, 10_000), st.integers(1, 4), st.integers(0, 4), st.integers(2, 12),
                  st.sampled_from([0.0, 0.5, 1.0, 2.0]), st.sampled_from([0.0, 0.3]))


@settings(max_examples=150, deadline=None)
@given(cases)
def test_outputs_are_well_formed(c):
    seed, B, K, V, T, mf = c
    t, d, toks, temps = _chain(seed, B, K, V, T, mf)
    o = oracle.verify_chain(t, d, toks, temps, seed, 3)
    for b in range(B):
        n = o["count"][b]
        assert 1 <= n <= K + 1
        assert (o["tokens"][b, :n - 1] == toks[b, :n - 1]).all()  # kept drafts, in order
        assert 0 <= o["tokens"][b, n - 1] < V
        assert (o["tokens"][b, n:] == -1).all()


@settings(max_examples=150, deadline=None)
@given(cases)
def test_chain_as_tree_is_the_chain(c):
    seed, B, K, V, T, mf = c
    if K == 0:
        return
    t, d, toks, temps = _chain(seed, B, K, V, T, mf)
    w = dict(kind="chain", target=t, draft=d, tokens=toks, temperature=temps, draft_kind=oracle.DRAFT_LOGITS,
             seed=seed, offset=5)
    tw = synth.chain_as_tree(w)
    a = oracle.verify_chain(t, d, toks, temps, seed, 5)
    b = oracle.verify_tree(tw["target"], tw["draft"], tw["node_tokens"], tw["parent"], tw["temperature"],
                           tw["max_depth"], seed, 5)
    assert (a["count"] == b["count"]).all()
    for r in range(B):
        n = a["count"][r]
        assert (a["tokens"][r, :n] == b["tokens"][r, :n]).all()


@settings(max_examples=100, deadline=None)
@given(cases)
def test_identical_distributions_accept_every_draft(c):
    seed, B, K, V, T, _ = c
    if T <= 0:
        return
    t, _, toks, temps = _chain(seed, B, K, V, T, 0.0)
    o = oracle.verify_chain(t, t[:, :K].copy(), toks, temps, seed, 1)
    assert (o["count"] == K + 1).all()


@settings(max_examples=100, deadline=None)
@given(cases)
def test_drafts_outside_the_target_support_are_rejected_at_once(c):
    seed, B, K, V, T, _ = c
    if T <= 0 or K == 0:
        return
    rng = np.random.default_rng(seed)
    t, d, toks, temps = _chain(seed, B, K, V, T, 0.0)
    half = V // 2
    t[:, :, half:] = -np.inf          # the target lives on [0, half)
    toks[:] = rng.integers(half, V, toks.shape)  # every draft outside it
    o = oracle.verify_chain(t, d, toks, temps, seed, 2)
    assert (o["count"] == 1).all()
    assert (o["tokens"][:, 0] < half).all()


@settings(max_examples=120, deadline=None)
@given(st.integers(0, 10_000), st.integers(1, 70))
def test_mask_is_the_ancestor_or_self_set(seed, N):
    """Any valid parent array (parent[i] in {-1} u [0, i)): bit j of row i is set iff j
    is i or an ancestor of i; depth is the number of nodes from the root's child down."""
    rng = np.random.default_rng(seed)
    par = np.array([[rng.integers(-1, i) if i else -1 for i in range(N)]], np.int32)
    o = oracle.tree_mask(par)
    assert o["valid"][0] == 1
    for i in range(N):
        anc, a = {i}, par[0, i]
        while a >= 0:
            anc.add(int(a))
            a = par[0, a]
        bits = {j for j in range(N) if (int(o["mask"][0, i, j // 32]) >> (j % 32)) & 1}
        assert bits == anc
        assert o["depth"][0, i] == len(anc)


@settings(max_examples=120, deadline=None)
@given(st.integers(0, 10_000), st.integers(2, 40), st.integers(1, 6))
def test_compaction_is_a_gather_from_the_original_cache(seed, N, D):
    """A root-to-node path (increasing node indices): rows base+d take the original rows
    base+path[d] for d < count-1; every other row is untouched."""
    rng = np.random.default_rng(seed)
    par = np.array([[rng.integers(-1, i) if i else -1 for i in range(N)]], np.int32)
    node = int(rng.integers(0, N))
    chain = []
    while node >= 0:
        chain.append(node)
        node = par[0, node]
    chain = chain[::-1][:D]
    path = np.full((1, D), -1, np.int32)
    path[0, :len(chain)] = chain
    count = np.array([len(chain) + 1], np.int32)
    R, rb = N + 8, 12
    base = np.array([int(rng.integers(0, R - N + 1))], np.int32)
    kv = rng.integers(0, 256, (1, R, rb), dtype=np.uint8)
    out = oracle.kv_compact(kv, path, count, base)
    want = kv.copy()
    for d, v in enumerate(chain):
        want[0, base[0] + d] = kv[0, base[0] + v]
    assert (out == want).all()
