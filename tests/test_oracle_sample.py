"""Pins of the oracle's draft sampling + verify (no GPU).

The drafted tokens are tied to numpy's own Philox4x64 (word 2 of block {k, row,
offset, 0}) and numpy's searchsorted on an fp64 softmax; greedy drafts to
numpy.argmax; the verify half to oracle.verify_chain given the same tokens; and
the whole round to the target law (the first emitted token of 2*10^5 rounds with
K = 1 against p_0, within the 99th percentile of an exact sampler's TV).
"""
import numpy as np

import oracle
from speculative_decoding_verification_53_gb300 import synth

GRID = 1 << 24


def _numpy_word2(k, row, offset, seed):
    val = k + (row << 64) + (offset << 128) - 1  # numpy advances the counter before a block
    val %= 1 << 256
    ctr = np.array([(val >> (64 * i)) & (2**64 - 1) for i in range(4)], np.uint64)
    blk = np.random.Philox(counter=ctr, key=np.array([seed, 0], np.uint64)).random_raw(4)
    return int(blk[2]) >> 40


def _softmax64(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def test_drafted_tokens_are_word2_inverse_cdf_draws_from_q():
    w = synth.tiny_chain(seed=12, V=50, K=4, B=30)
    seed, offset = 91, 6
    o = oracle.sample_and_verify(w["target"], w["draft"], w["temperature"], seed, offset)
    checked = 0
    for b in range(30):
        T = np.float64(np.float32(w["temperature"][b]))
        for k in range(4):
            q = _softmax64(w["draft"][b, k].astype(np.float64) / T)
            cdf = np.cumsum(q)
            t = _numpy_word2(k, b, offset, seed) / GRID * cdf[-1]
            expect = int(np.searchsorted(cdf, t, side="right"))
            if min(abs(cdf[expect] - t), abs(t - (cdf[expect - 1] if expect else 0.0))) > 1e-9:
                assert o["draft_tokens"][b, k] == expect
                checked += 1
    assert checked > 100


def test_greedy_rows_draft_the_argmax_and_the_verify_half_matches_verify_chain():
    w = synth.mixed_batch(seed=5, B=12, K=5, V=700)
    seed, offset = 4, 9
    draft = w["draft"]
    o = oracle.sample_and_verify(w["target"], draft, w["temperature"], seed, offset)
    d32 = synth.bf16_bits_to_f32(draft) if draft.dtype == np.uint16 else draft
    for b in range(12):
        if not w["temperature"][b] > 0:
            assert (o["draft_tokens"][b] == np.argmax(d32[b], axis=1)).all()
    v = oracle.verify_chain(w["target"], draft, o["draft_tokens"], w["temperature"], seed, offset,
                            draft_kind=oracle.DRAFT_LOGITS)
    for k in ("tokens", "count", "accept_prob"):
        np.testing.assert_array_equal(o[k], v[k])
    assert (o["margin"] <= v["margin"]).all()


def test_invalid_draft_row_invalidates_the_round():
    w = synth.tiny_chain(seed=13, V=32, K=3, B=3)
    d = w["draft"].copy()
    d[1, 2, 5] = np.nan
    o = oracle.sample_and_verify(w["target"], d, w["temperature"], 1, 1)
    assert o["draft_tokens"][1, 2] == -1 and o["count"][1] == 0 and (o["tokens"][1] == -1).all()
    assert (o["count"][[0, 2]] >= 1).all()


def test_round_law_is_the_target_law():
    """K = 1, V = 8: draft sampled inside the call; the first emitted token follows p_0."""
    rng = np.random.default_rng(17)
    V, n = 8, 200000
    t = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    d = (t[:1] + rng.normal(0, 1.0, (1, V))).astype(np.float32)
    o = oracle.sample_and_verify(np.broadcast_to(t, (n, 2, V)).copy(), np.broadcast_to(d, (n, 1, V)).copy(),
                                 np.ones(n, np.float32), 123, 0)
    p0 = _softmax64(t[0])
    tv = 0.5 * np.abs(np.bincount(o["tokens"][:, 0], minlength=V) / n - p0).sum()
    exact = [0.5 * np.abs(rng.multinomial(n, p0) / n - p0).sum() for _ in range(300)]
    assert tv <= np.quantile(exact, 0.99), tv
    q = _softmax64(d[0])
    tvq = 0.5 * np.abs(np.bincount(o["draft_tokens"][:, 0], minlength=V) / n - q).sum()
    assert tvq <= np.quantile([0.5 * np.abs(rng.multinomial(n, q) / n - q).sum() for _ in range(300)], 0.99)
