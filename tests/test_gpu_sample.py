"""GPU parity of spec_sample_and_verify (draft tokens drawn on the GPU, then verified).

Drafted tokens, emitted tokens and counts must equal the oracle's on the same seeded
inputs, except on rows where the oracle saw a decision (a draft draw included)
within 1e-5 of its boundary; a 10^6-round run checks the target law end to end.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth
from _harness import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_53_gb300 import build
    build.build()
    import speculative_decoding_verification_53_gb300 as m
    m.lib()
    return m


def _gpu(sv, w, seed, offset, **kw):
    import torch
    xd, ot, oc, ap = sv.spec_sample_and_verify(to_dev(w["target"]), to_dev(w["draft"]),
                                               to_dev(w["temperature"].astype(np.float32)), seed, offset,
                                               want_accept_prob=True, **kw)
    torch.cuda.synchronize()
    return dict(draft_tokens=xd.cpu().numpy(), tokens=ot.cpu().numpy(), count=oc.cpu().numpy(),
                accept_prob=ap.cpu().numpy())


@pytest.mark.parametrize("case", ["mixed", "tiny_fp32", "vocab128k", "k0", "k1_many_rows"])
def test_sample_and_verify_matches_oracle(sv, case):
    if case == "mixed":
        w = synth.mixed_batch(seed=81, B=24, K=5, V=32000)
    elif case == "tiny_fp32":
        w = synth.tiny_chain(seed=82, V=1024, K=4, B=16)
    elif case == "vocab128k":
        w = synth.large_batch(seed=83, temperature=0.8, sigma=1.0, B=4, K=5, V=128256)
    elif case == "k0":
        w = synth.tiny_chain(seed=84, V=3000, K=0, B=3)
    else:
        w = synth.tiny_chain(seed=85, V=500, K=1, B=700)
    for seed, offset in [(3, 0), (3, 1)]:
        g = _gpu(sv, w, seed, offset)
        o = oracle.sample_and_verify(w["target"], w["draft"], w["temperature"], seed, offset)
        compare(g, o, keys=("draft_tokens", "tokens", "count"))


def test_sample_and_verify_without_workspace_and_invalid_rows(sv):
    w = synth.tiny_chain(seed=86, V=2048, K=3, B=6)
    d = w["draft"].copy()
    d[2, 1, 100] = np.nan
    d[4, 0, :] = -np.inf
    w = dict(w, draft=d)
    g = _gpu(sv, w, 9, 2, workspace=None)
    o = oracle.sample_and_verify(w["target"], w["draft"], w["temperature"], 9, 2)
    assert g["count"][2] == 0 and g["count"][4] == 0
    assert g["draft_tokens"][2, 1] == -1 and g["draft_tokens"][4, 0] == -1
    compare(g, o, keys=("draft_tokens", "tokens", "count"))


def test_sample_and_verify_law(sv):
    """K = 1, V = 8, 10^6 rounds: the drafted token follows q_0 and the first emitted
    token p_0 (TV within the 99th percentile of an exact sampler's TV)."""
    import torch
    V, B, calls = 8, 62500, 16
    rng = np.random.default_rng(47)
    t = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    d = (t[:1] + rng.normal(0, 1.0, (1, V))).astype(np.float32)
    tt = to_dev(np.broadcast_to(t, (B, 2, V)).copy())
    dd = to_dev(np.broadcast_to(d, (B, 1, V)).copy())
    temps = torch.ones(B, device="cuda")
    first, drafted = [], []
    for c in range(calls):
        xd, ot, _, _ = sv.spec_sample_and_verify(tt, dd, temps, 500 + c, c)
        first.append(ot[:, 0].cpu().numpy())
        drafted.append(xd[:, 0].cpu().numpy())
    n = B * calls

    def sm(z):
        e = np.exp(z.astype(np.float64) - z.max())
        return e / e.sum()

    for got, law in ((np.concatenate(first), sm(t[0])), (np.concatenate(drafted), sm(d[0]))):
        tv = 0.5 * np.abs(np.bincount(got, minlength=V) / n - law).sum()
        exact = [0.5 * np.abs(rng.multinomial(n, law) / n - law).sum() for _ in range(300)]
        assert tv <= np.quantile(exact, 0.99), tv


def test_sample_and_verify_bad_arguments(sv):
    import ctypes
    lib = sv.lib()
    vp = ctypes.c_void_p(16)
    f = lib.spec_sample_and_verify
    assert f(vp, 0, vp, 0, vp, 1, 65, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert f(vp, 0, None, 0, vp, 1, 3, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert f(vp, 3, vp, 0, vp, 1, 3, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert f(None, 0, None, 0, None, 0, 3, 100, 0, 0, None, None, None, None, None, 0, None) == sv.SV_OK


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_sample_and_verify_largest_vocabulary(sv, dt):
    """V = 2^24, the largest vocabulary the boundary takes: the draft rows are too long to
    stage, so the streaming sampler draws from them with a cluster wide enough for its
    tile sums; a sampling row and a greedy row against the oracle."""
    w = synth.tiny_chain(seed=87, V=1 << 24, K=1, B=2)
    w["temperature"] = np.array([1.0, 0.0], np.float32)
    if dt == "bf16":
        w["target"] = synth.f32_to_bf16_bits(w["target"])
        w["draft"] = synth.f32_to_bf16_bits(w["draft"])
    g = _gpu(sv, w, 5, 1)
    o = oracle.sample_and_verify(w["target"], w["draft"], w["temperature"], 5, 1)
    assert compare(g, o, keys=("draft_tokens", "tokens", "count")) <= 1


def test_sample_and_verify_longest_draft(sv):
    """K = 64 drafted positions, the most the boundary takes, sampling and greedy rows."""
    w = synth.tiny_chain(seed=88, V=300, K=64, B=6, sigma=0.05)
    w["temperature"][::2] = 0.0
    for seed, offset in [(7, 0), (7, 3)]:
        g = _gpu(sv, w, seed, offset)
        o = oracle.sample_and_verify(w["target"], w["draft"], w["temperature"], seed, offset)
        assert compare(g, o, keys=("draft_tokens", "tokens", "count")) <= 1
