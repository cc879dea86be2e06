"""GPU parity: the CUDA library against the fp64 oracle on the same seeded inputs.

Covers the five verify workloads (tiny fp32 chain, single-stream V=128256 with
draft probabilities, mixed greedy/sampling batch, draft trees, large batch
V=152064 at three temperatures), ragged and misaligned vocabularies, and the
degenerate cases (K=0, V=1, ties, masked and invalid rows).
"""
import ctypes

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth
from _harness import compare, gpu_chain, gpu_tree, oracle_chain, oracle_tree, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_53_gb300 import build
    build.build()


# ---------------------------------------------------------------- chains

def test_tiny_chain_rounds_seeded_by_round():
    """fp32, B=1, K=4, V=1024 and V=8: round s uses seed s for inputs and Philox."""
    excused = 0
    for V in (1024, 8):
        for s in range(60):
            w = synth.tiny_chain(seed=s, V=V)
            excused += compare(gpu_chain(w, seed=s), oracle_chain(w, seed=s))
    assert excused <= 2


@pytest.mark.parametrize("B,V,T", [(4096, 1024, 1.0), (300, 4099, 0.6), (64, 50000, 1.3)])
def test_tiny_chain_batched(B, V, T):
    w = synth.tiny_chain(seed=B + V, V=V, B=B, temperature=T)
    assert compare(gpu_chain(w, seed=11, offset=5), oracle_chain(w, seed=11, offset=5)) <= max(2, B // 500)


def test_single_stream_full_size_rounds():
    """bf16 target V=128256, K=5, fp32 draft probabilities, T=0.8, B=1 per call."""
    excused = 0
    w0 = synth.single_stream(seed=0, B=12)
    for s in range(12):
        w = {k: (v[s:s + 1] if isinstance(v, np.ndarray) else v) for k, v in w0.items()}
        excused += compare(gpu_chain(w, seed=s, offset=s), oracle_chain(w, seed=s, offset=s))
    assert excused <= 1


def test_mixed_batch_full_size():
    """B=64, K=5, V=32000 bf16; even rows greedy, odd rows T=1; sigma by row."""
    w = synth.mixed_batch(seed=3)
    g, o = gpu_chain(w, seed=3), oracle_chain(w, seed=3)
    assert compare(g, o) <= 1
    greedy = w["temperature"] <= 0
    assert np.array_equal(g["tokens"][greedy], o["tokens"][greedy])  # greedy rows are exact


@pytest.mark.parametrize("B,V", [(200, 40008), (160, 16392), (160, 152064)])
def test_staged_walk_one_slot(B, V):
    """Batches past one CTA per SM take the staged walk with a single slot (the next
    position's chunk copied only once the current one is decided, warmed in L2 for
    large chunks): ragged last CTAs, greedy and sampling rows, bf16 target and draft
    logits."""
    w = synth.mixed_batch(seed=B + V, B=B, K=4, V=V)
    g, o = gpu_chain(w, seed=7, offset=2), oracle_chain(w, seed=7, offset=2)
    assert compare(g, o) <= max(1, B // 200)
    greedy = w["temperature"] <= 0
    assert np.array_equal(g["tokens"][greedy], o["tokens"][greedy])


@pytest.mark.parametrize("tdt,ddt", [("f32", "bf16"), ("bf16", "f32"), ("f32", "f32")])
def test_staged_walk_one_slot_fp32_rows(tdt, ddt):
    """The single-slot walk with fp32 target or draft-logit rows: the draft row is reduced
    from global memory (fp32 loads) and re-read for the draw, the target staged."""
    w = synth.mixed_batch(seed=61, B=160, K=3, V=16392)
    if tdt == "f32":
        w["target"] = synth.bf16_bits_to_f32(w["target"])
    if ddt == "f32":
        w["draft"] = synth.bf16_bits_to_f32(w["draft"])
    g, o = gpu_chain(w, seed=5, offset=1), oracle_chain(w, seed=5, offset=1)
    assert compare(g, o) <= 1
    greedy = w["temperature"] <= 0
    assert np.array_equal(g["tokens"][greedy], o["tokens"][greedy])


def test_moderate_batch_position_parallel_with_bad_rows():
    """B = 32, V = 32000: the automatic path runs the position-parallel kernel in
    clusters of 2 over two waves.  Rows carry NaN, +inf, all -inf or an out-of-range
    token at various positions; only data the rule reads may invalidate a row."""
    w = synth.mixed_batch(seed=77, B=32, K=5, V=32000)
    t, d, toks = w["target"].copy(), w["draft"].copy(), w["tokens"].copy()
    nan, inf, ninf = np.uint16(0x7FC0), np.uint16(0x7F80), np.uint16(0xFF80)  # bf16 bit patterns
    t[0, 0, 11] = nan
    t[1, 3, 5] = inf
    t[2, 5, :] = ninf
    d[3, 1, 7] = nan
    toks[4, 2] = 32000
    toks[5, 0] = -3
    t[6, 2, :16000] = ninf  # half masked: still valid
    w2 = dict(w, target=t, draft=d, tokens=toks)
    g, o = gpu_chain(w2, seed=5, offset=1), oracle_chain(w2, seed=5, offset=1)
    assert compare(g, o) <= 1
    assert g["count"][4] == 0 and g["count"][5] == 0 and g["count"][0] == 0


@pytest.fixture(scope="module")
def large_batch_sigma1():
    return synth.large_batch(seed=5, temperature=0.7, sigma=1.0)


@pytest.mark.parametrize("T", [0.0, 0.7, 1.5])
def test_large_batch_full_size_sampled_rows(large_batch_sigma1, T):
    """B=256, K=8, V=152064 bf16 target and draft logits: the full batch runs on the GPU
    in the benchmark's launch shape; 24 sampled rows are recomputed by the oracle."""
    w = synth.redraw_tokens(large_batch_sigma1, T, seed=int(T * 10) + 1)
    rows = np.random.default_rng(int(T * 100)).choice(256, 24, replace=False)
    g = gpu_chain(w, seed=77, offset=int(T * 10))
    o = oracle_chain(w, seed=77, offset=int(T * 10), rows=rows)
    assert compare(g, o, rows=rows) <= 1
    assert (g["count"] >= 1).all() and (g["count"] <= 9).all()


def test_large_batch_collapse_sigma3():
    """T=1.5 with draft noise sigma=3: acceptance collapses, rounds emit ~1 token."""
    w = synth.large_batch(seed=9, temperature=1.5, sigma=3.0, B=64)
    rows = np.arange(0, 64, 4)
    g = gpu_chain(w, seed=1)
    assert compare(g, oracle_chain(w, seed=1, rows=rows), rows=rows) <= 1
    assert g["count"].mean() < 1.6


# ----------------------------------------------------------------- trees

@pytest.fixture(scope="module")
def tree_workload():
    return synth.tree(seed=4)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_full_size(tree_workload, T):
    """B=16, N=60, depth <= 6, V=128256 bf16; greedy and sampling at T=1."""
    w = dict(tree_workload)
    w["temperature"] = np.full(16, T, np.float32)
    g, o = gpu_tree(w, seed=8), oracle_tree(w, seed=8)
    assert compare(g, o, keys=("tokens", "count", "path")) <= 1


def test_chain_as_tree_matches_oracle_chain():
    w = synth.tiny_chain(seed=12, V=3001, K=5, B=200, temperature=0.9)
    tw = synth.chain_as_tree(w)
    oc = oracle_chain(w, seed=2, offset=3)
    gt = gpu_tree(tw, seed=2, offset=3)
    n = compare({"tokens": gt["tokens"], "count": gt["count"]}, oc)
    assert n <= 1


def test_tree_small_random_shapes():
    rng = np.random.default_rng(0)
    B, N, V = 40, 24, 3000
    target = rng.normal(0, 2, (B, N + 1, V)).astype(np.float32)
    draft = (target + rng.normal(0, 1, (B, N + 1, V))).astype(np.float32)
    par = np.empty((B, N), np.int32)
    toks = np.empty((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            par[b, i] = rng.integers(-1, min(i, 4)) if i else -1
        toks[b] = rng.integers(0, V, N)
        # make some children likely under p: copy the draft argmax of the parent row
        for i in range(N):
            if rng.random() < 0.5:
                toks[b, i] = int(np.argmax(draft[b, par[b, i] + 1]))
    depth = np.zeros((B, N), int)
    for b in range(B):
        for i in range(N):
            depth[b, i] = 1 if par[b, i] < 0 else depth[b, par[b, i]] + 1
    for T in (0.0, 1.0):
        w = dict(kind="tree", target=target, draft=draft, draft_kind=oracle.DRAFT_LOGITS, node_tokens=toks,
                 parent=par, temperature=np.full(B, T, np.float32), max_depth=int(depth.max()), seed=1, offset=0)
        assert compare(gpu_tree(w), oracle_tree(w), keys=("tokens", "count", "path")) <= 1
    wp = dict(w)
    wp["draft_kind"] = oracle.DRAFT_PROBS
    e = np.exp(draft - draft.max(2, keepdims=True))
    wp["draft"] = (e / e.sum(2, keepdims=True)).astype(np.float32)
    assert compare(gpu_tree(wp), oracle_tree(wp), keys=("tokens", "count", "path")) <= 1


def test_tree_at_the_node_and_depth_limits():
    """N = 1024 nodes (16 chains of 64 under the root, so depth 64 = max_depth): the walk
    may descend 64 levels; greedy and sampling against the oracle, draft as logits."""
    rng = np.random.default_rng(5)
    B, N, V, D = 2, 1024, 2048, 64
    target = rng.normal(0, 2, (B, N + 1, V)).astype(np.float32)
    draft = (target + rng.normal(0, 0.3, (B, N + 1, V))).astype(np.float32)
    par = np.array([i - 16 if i >= 16 else -1 for i in range(N)], np.int32)
    par = np.tile(par, (B, 1))
    toks = rng.integers(0, V, (B, N)).astype(np.int32)
    for b in range(B):  # most nodes carry the target's argmax of their parent's row: long accepted paths
        for i in range(N):
            if rng.random() < 0.97:
                toks[b, i] = int(np.argmax(target[b, par[b, i] + 1]))
    for T in (0.0, 1.0):
        w = dict(kind="tree", target=target, draft=draft, draft_kind=oracle.DRAFT_LOGITS, node_tokens=toks,
                 parent=par, temperature=np.full(B, T, np.float32), max_depth=D, seed=2, offset=0)
        g, o = gpu_tree(w), oracle_tree(w)
        assert compare(g, o, keys=("tokens", "count", "path")) <= 1
        if T == 0.0:
            assert o["count"].min() > 8  # greedy walks go deep


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("V", [1, 7, 9, 255, 1001, 4097, 33001])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ragged_and_misaligned_vocab(V, dt):
    w = synth.tiny_chain(seed=V, V=V, K=3, B=37, temperature=0.8)
    if dt == "bf16":
        w["target"] = synth.f32_to_bf16_bits(w["target"])
        w["draft"] = synth.f32_to_bf16_bits(w["draft"])
    assert compare(gpu_chain(w), oracle_chain(w)) <= 1
    wg = dict(w)
    wg["temperature"] = np.zeros(37, np.float32)
    assert compare(gpu_chain(wg), oracle_chain(wg)) == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_largest_vocabulary(dt):
    """V = 2^24, the largest vocabulary the boundary takes: a chunk per CTA far beyond shared
    memory, so the rows are streamed; greedy and sampling rows against the oracle.  One more
    element is refused before anything runs."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    V = 1 << 24
    w = synth.tiny_chain(seed=91, V=V, K=1, B=2, temperature=1.0)
    w["temperature"] = np.array([1.0, 0.0], np.float32)  # a sampling row and a greedy row
    if dt == "bf16":
        w["target"] = synth.f32_to_bf16_bits(w["target"])
        w["draft"] = synth.f32_to_bf16_bits(w["draft"])
    assert compare(gpu_chain(w, seed=4, offset=1), oracle_chain(w, seed=4, offset=1)) <= 1
    t = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    st = sv.lib().spec_verify_chain(ctypes.c_void_p(t.data_ptr()), 0, ctypes.c_void_p(t.data_ptr()), 0, 1,
                                    ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(t.data_ptr()), 1, 1, V + 1, 0, 0,
                                    ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(t.data_ptr()), None, None, 0, None)
    assert st == sv.SV_ERR_INVALID_ARG


def test_largest_batch():
    """B = 65535, the most batch rows the boundary takes: a chain with greedy and sampling
    rows, and a two-level tree per row, against the oracle at a small vocabulary; one row
    more is refused before anything runs."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    B = 65535
    w = synth.tiny_chain(seed=77, V=64, K=2, B=B, temperature=0.9)
    w["temperature"][::3] = 0.0
    assert compare(gpu_chain(w, seed=9, offset=2), oracle_chain(w, seed=9, offset=2)) <= B // 2000
    rng = np.random.default_rng(8)
    N, V = 3, 32
    target = rng.normal(0, 2, (B, N + 1, V)).astype(np.float32)
    draft = (target + rng.normal(0, 1, (B, N + 1, V))).astype(np.float32)
    par = np.tile(np.array([-1, 0, -1], np.int32), (B, 1))  # root -> {0 -> 1, 2}
    toks = rng.integers(0, V, (B, N)).astype(np.int32)
    temp = np.where(np.arange(B) % 4 == 0, 0.0, 1.0).astype(np.float32)
    wt = dict(kind="tree", target=target, draft=draft, draft_kind=oracle.DRAFT_LOGITS, node_tokens=toks,
              parent=par, temperature=temp, max_depth=2, seed=6, offset=0)
    assert compare(gpu_tree(wt), oracle_tree(wt), keys=("tokens", "count", "path")) <= B // 2000
    t = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    st = sv.lib().spec_verify_chain(p, 0, p, 0, 1, p, p, B + 1, 1, 8, 0, 0, p, p, None, None, 0, None)
    assert st == sv.SV_ERR_INVALID_ARG


@pytest.mark.parametrize("K", [0, 1, 2, 64])
def test_draft_length_extremes(K):
    w = synth.tiny_chain(seed=K, V=513, K=K, B=20, temperature=1.0, sigma=0.2)
    assert compare(gpu_chain(w), oracle_chain(w)) <= 1


def test_position_parallel_at_its_26_position_limit():
    """K = 25 puts 26 positions into the position-parallel kernel's packed arrival word
    (reject bits 11..36, invalid bits 37..62; B = 1 with aligned rows takes that kernel).
    Near-certain acceptance reaches the last positions; a NaN in the bonus row makes
    exactly the rounds that reach it invalid.  K = 26 is past the limit and walks."""
    for K in (25, 26):
        excused = 0
        for s in range(8):
            w = synth.tiny_chain(seed=100 + s, V=1024, K=K, B=1, temperature=1.0, sigma=0.05)
            if s >= 4:
                t = w["target"].copy()
                t[0, K, 7] = np.nan
                w = dict(w, target=t)
            g, o = gpu_chain(w, seed=s, offset=s), oracle_chain(w, seed=s, offset=s)
            excused += compare(g, o)
        assert excused <= 1


def test_greedy_ties_and_entry_point():
    import speculative_decoding_verification_53_gb300 as sv
    rng = np.random.default_rng(8)
    B, K, V = 200, 5, 3000
    vals = rng.integers(-2, 2, (B, K + 1, V)).astype(np.float32)  # heavy ties
    target = synth.f32_to_bf16_bits(vals)
    am = np.argmax(vals, axis=2)
    toks = am[:, :K].astype(np.int32).copy()
    cut = rng.integers(0, K + 1, B)
    for b in range(B):
        if cut[b] < K:
            toks[b, cut[b]] = (am[b, cut[b]] + 1) % V
    o = oracle.greedy_accept(target, toks)
    ot, oc = sv.spec_greedy_accept(to_dev(target), to_dev(toks))
    assert np.array_equal(ot.cpu().numpy(), o["tokens"]) and np.array_equal(oc.cpu().numpy(), o["count"])


def test_identical_distributions_accept_everything():
    w = synth.tiny_chain(seed=1, V=2000, K=6, B=64)
    w["draft"] = w["target"][:, :6].copy()
    g = gpu_chain(w)
    assert (g["count"] == 7).all()
    assert compare(g, oracle_chain(w)) == 0


def test_masked_invalid_and_zero_q_rows():
    w = synth.tiny_chain(seed=2, V=700, K=3, B=12)
    t, toks = w["target"].copy(), w["tokens"].copy()
    t[0, 0, 3] = np.nan
    t[1, 0, :] = -np.inf
    t[2, 0, 5] = np.inf
    toks[3, 2] = 700
    toks[4, 0] = -1
    t[5, :, :350] = -np.inf  # masked half: valid
    w2 = dict(w, target=t, tokens=toks)
    g, o = gpu_chain(w2), oracle_chain(w2)
    assert g["count"][:5].tolist() == [0, 0, 0, 0, 0]
    assert compare(g, o) == 0
    # draft probabilities with q(x) = 0 at the drafted token: accepted iff p(x) > 0
    wp = synth.single_stream(seed=3, V=900, K=3, B=16)
    wp["draft"][:, :, :] = 0.0
    wp["draft"][np.arange(16)[:, None], np.arange(3)[None, :], (wp["tokens"] + 1) % 900] = 1.0
    g, o = gpu_chain(wp), oracle_chain(wp)
    assert compare(g, o) == 0
    assert (g["count"] == 4).all()


def test_count_invalid_rows_status():
    """spec_verify_count_invalid counts the rows with count 0; rows_status turns a
    non-zero count into SV_ERR_BAD_INPUT."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    w = synth.tiny_chain(seed=2, V=700, K=3, B=12)
    t = w["target"].copy()
    t[0, 0, 3] = np.nan
    t[1, 0, :] = -np.inf
    g = gpu_chain(dict(w, target=t))
    cnt = torch.from_numpy(g["count"]).cuda()
    assert int(sv.spec_verify_count_invalid(cnt).item()) == int((g["count"] == 0).sum()) == 2
    assert sv.rows_status(cnt) == sv.SV_ERR_BAD_INPUT
    assert sv.rows_status(torch.from_numpy(gpu_chain(w)["count"]).cuda()) == sv.SV_OK
    rng = np.random.default_rng(4)
    for B in (0, 1, 1023, 1024, 1025, 300001):
        c = rng.integers(0, 3, B).astype(np.int32)
        got = sv.spec_verify_count_invalid(torch.from_numpy(c).cuda()) if B else \
            sv.spec_verify_count_invalid(torch.zeros(0, dtype=torch.int32, device="cuda"))
        assert int(got.item()) == int((c == 0).sum())


def _bad_after_first_rejection():
    """Rows whose first draft is surely rejected (p(x_0) = 0, or x_0 != argmax on greedy
    rows) carry invalid data only at later positions, which the rule never reads."""
    w = synth.tiny_chain(seed=6, V=640, K=4, B=6)
    t, d, toks = w["target"].copy(), w["draft"].copy(), w["tokens"].copy()
    temp = w["temperature"].copy()
    for b in range(6):
        t[b, 0, toks[b, 0]] = -np.inf          # p_0(x_0) = 0: rejected at position 0
    t[0, 2, 7] = np.nan
    t[1, 3, :] = -np.inf
    t[2, 4, 9] = np.inf
    d[3, 2, 11] = np.nan                       # draft logits invalid at position 2
    temp[4:] = 0.0                             # greedy rows: x_0 is not the argmax (its logit is -inf)
    t[4, 1, 3] = np.nan
    t[5, 4, :] = -np.inf
    return dict(w, target=t, draft=d, tokens=toks, temperature=temp)


def test_invalid_rows_after_the_first_rejection_are_ignored():
    w = _bad_after_first_rejection()
    g, o = gpu_chain(w), oracle_chain(w)
    assert (o["count"] == 1).all()
    assert compare(g, o) == 0
    assert (g["count"] == 1).all()


def test_empty_batch_is_a_noop():
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    t = torch.zeros((0, 3, 100), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((0, 2, 100), dtype=torch.bfloat16, device="cuda")
    ot, oc, _ = sv.spec_verify_chain(t, d, torch.zeros((0, 2), dtype=torch.int32, device="cuda"),
                                     torch.zeros((0,), device="cuda"), 0, 0, draft_kind="logits")
    assert ot.shape == (0, 3) and oc.shape == (0,)


def test_bad_arguments_raise():
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    t = torch.zeros((2, 3, 100), dtype=torch.float32, device="cuda")
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_tree(torch.zeros((1, 2, 10), device="cuda"), torch.zeros((1, 2, 10), device="cuda"),
                            torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                            torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                            torch.ones(1, device="cuda"), 0, 0, 0, draft_kind="logits")
    with pytest.raises(ValueError):
        sv.spec_verify_chain(t, torch.zeros((2, 3, 100), device="cuda"),
                             torch.zeros((2, 2), dtype=torch.int32, device="cuda"), torch.ones(2, device="cuda"),
                             0, 0, draft_kind="logits")


# ------------------------------------------------------ multi-draft siblings

@pytest.mark.parametrize("rule", [oracle.SIBLINGS_IID, oracle.SIBLINGS_WOR])
def test_tree_iid_children_both_rules_full_size(rule):
    """Trees whose children were drafted i.i.d. from q (tokens may repeat among siblings),
    V=128256, verified under either sibling rule, against the oracle under the same rule."""
    w = synth.redraw_children_iid(synth.tree(seed=71, temperature=1.0, B=8), seed=3)
    compare(gpu_tree(w, seed=5, sibling_rule=rule), oracle_tree(w, seed=5, sibling_rule=rule),
            keys=("tokens", "count", "path"))


def test_gpu_multidraft_law_with_iid_children():
    """10^6 rounds of a root with three children drawn i.i.d. from q (V=16): with the i.i.d.
    rule the first emitted token follows p (TV within the 99th percentile of an exact
    sampler's TV); the without-replacement rule on the same drafts is visibly biased."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    V, C, B, calls = 16, 3, 62500, 16
    rng = np.random.default_rng(43)
    t = (rng.normal(0, 0.8, (C + 1, V))).astype(np.float32)
    d = (t + rng.normal(0, 0.8, (C + 1, V))).astype(np.float32)
    q = np.exp(d[0].astype(np.float64) - d[0].max())
    q /= q.sum()
    p = np.exp(t[0].astype(np.float64) - t[0].max())
    p /= p.sum()
    tt = to_dev(np.broadcast_to(t, (B, C + 1, V)).copy())
    dd = to_dev(np.broadcast_to(d, (B, C + 1, V)).copy())
    par = to_dev(np.full((B, C), -1, np.int32))
    temps = torch.ones(B, device="cuda")
    first = {"iid": [], "without_replacement": []}
    for c in range(calls):
        toks = to_dev(rng.choice(V, (B, C), p=q).astype(np.int32))
        for rule in first:
            ot, _, _ = sv.spec_verify_tree(tt, dd, toks, par, temps, 1, 2000 + c, c, draft_kind="logits",
                                           sibling_rule=rule)
            first[rule].append(ot[:, 0].cpu().numpy())
    n = B * calls
    exact = [0.5 * np.abs(rng.multinomial(n, p) / n - p).sum() for _ in range(300)]
    tv = {r: 0.5 * np.abs(np.bincount(np.concatenate(v), minlength=V) / n - p).sum() for r, v in first.items()}
    assert tv["iid"] <= np.quantile(exact, 0.99), tv
    assert tv["without_replacement"] > 2 * np.quantile(exact, 0.99), tv


# ----------------------------------------------------------- statistics

def test_gpu_output_law_and_expected_count():
    """10^6 rounds (V=8, K=4): the first emitted token follows p_0 (TV within the 99th
    percentile of an exact sampler's TV), E[count] = sum_j prod_{i<j} alpha_i."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    V, K, B, calls = 8, 4, 62500, 16
    rng = np.random.default_rng(41)
    t = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    d = (t[:K] + rng.normal(0, 0.5, (K, V))).astype(np.float32)
    qs = np.exp(d - d.max(1, keepdims=True))
    qs /= qs.sum(1, keepdims=True)
    tt = to_dev(np.broadcast_to(t, (B, K + 1, V)).copy())
    dd = to_dev(np.broadcast_to(d, (B, K, V)).copy())
    temps = torch.ones(B, device="cuda")
    first, counts = [], []
    for c in range(calls):
        toks = np.stack([rng.choice(V, B, p=qs[k]) for k in range(K)], 1).astype(np.int32)
        ot, oc, _ = sv.spec_verify_chain(tt, dd, to_dev(toks), temps, 1000 + c, c, draft_kind="logits")
        first.append(ot[:, 0].cpu().numpy())
        counts.append(oc.cpu().numpy())
    first, counts = np.concatenate(first), np.concatenate(counts).astype(np.float64)
    n = first.size
    p0 = np.exp(t[0] - t[0].max()).astype(np.float64)
    p0 /= p0.sum()
    tv = 0.5 * np.abs(np.bincount(first, minlength=V) / n - p0).sum()
    exact = [0.5 * np.abs(rng.multinomial(n, p0) / n - p0).sum() for _ in range(300)]
    assert tv <= np.quantile(exact, 0.99), tv
    assert tv < 0.01
    p = [np.exp(t[i] - t[i].max()) / np.exp(t[i] - t[i].max()).sum() for i in range(K)]
    alphas = [np.minimum(p[i], qs[i]).sum() for i in range(K)]
    expect = sum(np.prod(alphas[:j]) for j in range(K + 1))
    assert abs(counts.mean() - expect) < 4 * counts.std() / np.sqrt(n)
