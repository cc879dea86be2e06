"""The seeded input generators follow the stated recipes (no GPU, small sizes).

They hold none of the method's arithmetic; these checks make sure the parity tests
and the bench run on the workloads described: shapes and dtypes, temperatures, the
per-row draft noise, the Zipf prior, probabilities that sum to one, tree structure
and accepted paths.
"""
import numpy as np

from speculative_decoding_verification_53_gb300 import synth


def _softmax(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def test_single_stream_recipe():
    w = synth.single_stream(seed=3, V=4000, B=3)
    assert w["target"].shape == (3, 6, 4000) and w["target"].dtype == np.uint16  # bf16 bit patterns
    assert w["draft"].shape == (3, 5, 4000) and w["draft"].dtype == np.float32
    np.testing.assert_allclose(w["draft"].sum(axis=2), 1.0, atol=1e-5)  # draft probabilities
    assert (w["temperature"] == np.float32(0.8)).all()
    assert w["tokens"].shape == (3, 5) and ((w["tokens"] >= 0) & (w["tokens"] < 4000)).all()
    t = synth.bf16_bits_to_f32(w["target"]).astype(np.float64)
    # the Zipf(1.1) prior: mean logit falls by 1.1 ln(ratio) between id bands
    lo, hi = t[..., 10:20].mean(), t[..., 3000:4000].mean()
    expect = -1.1 * (np.log(np.arange(3001, 4001)).mean() - np.log(np.arange(11, 21)).mean())
    assert abs((hi - lo) - expect) < 0.6


def test_mixed_batch_recipe():
    w = synth.mixed_batch(seed=5, B=12, K=5, V=6000)
    assert w["target"].dtype == np.uint16 and w["draft"].dtype == np.uint16
    temps = w["temperature"]
    assert (temps[0::2] == 0).all() and (temps[1::2] == 1).all()  # even rows greedy, odd rows T = 1
    t = synth.bf16_bits_to_f32(w["target"]).astype(np.float64)
    d = synth.bf16_bits_to_f32(w["draft"]).astype(np.float64)
    assert abs(t.std() - 2.0) < 0.1
    for b in range(12):
        sigma = (0.25, 1.0, 4.0)[b % 3]
        assert abs((d[b] - t[b, :5]).std() / sigma - 1) < 0.1
        if temps[b] <= 0:  # greedy rows draft the argmax of the draft logits
            assert (w["tokens"][b] == d[b].argmax(axis=1)).all()


def test_large_batch_recipe():
    w = synth.large_batch(seed=7, temperature=1.5, sigma=3.0, B=4, V=8192)
    assert w["target"].shape == (4, 9, 8192) and w["draft"].shape == (4, 8, 8192)
    assert (w["temperature"] == np.float32(1.5)).all()
    t = synth.bf16_bits_to_f32(w["target"]).astype(np.float64)
    d = synth.bf16_bits_to_f32(w["draft"]).astype(np.float64)
    assert abs((d - t[:, :8]).std() / 3.0 - 1) < 0.05


def test_tree_recipe():
    w = synth.tree(seed=9, B=2, N=60, V=3000)
    par, tok = w["parent"], w["node_tokens"]
    assert par.shape == (2, 60) and w["target"].shape == (2, 61, 3000) and w["draft"].shape == (2, 61, 3000)
    d = synth.bf16_bits_to_f32(w["draft"])
    for b in range(2):
        depth = np.zeros(60, int)
        for i in range(60):
            p = par[b, i]
            assert -1 <= p < i  # parents come before their children
            depth[i] = 1 if p < 0 else depth[p] + 1
        assert depth.max() <= w["max_depth"]
        for p in range(-1, 60):
            kids = np.flatnonzero(par[b] == p)
            assert len(kids) <= 3
            q = _softmax(d[b, 0 if p < 0 else p + 1])  # the row the children were proposed from
            qk = q[tok[b, kids]]
            assert (np.diff(qk) <= 1e-12).all()  # siblings by descending draft probability
            assert len(set(tok[b, kids])) == len(kids)  # without replacement
            if len(kids):
                assert set(tok[b, kids]) == set(np.argsort(-q, kind="stable")[:len(kids)])  # the top ones


def test_iid_redraw_keeps_the_tree_and_draws_from_the_parents_q():
    w = synth.tree(seed=11, B=1, N=60, V=40)
    r = synth.redraw_children_iid(w, seed=4)
    assert (r["parent"] == w["parent"]).all()
    assert ((r["node_tokens"] >= 0) & (r["node_tokens"] < 40)).all()
    assert (r["node_tokens"] != w["node_tokens"]).any()


def test_random_parents_shapes():
    for shape in ("bfs", "random", "chain", "star"):
        par = synth.random_parents(13, 3, 50, shape=shape, max_depth=8)
        assert par.shape == (3, 50)
        i = np.arange(50)
        assert ((par >= -1) & (par < i)).all()
    assert (synth.random_parents(13, 2, 20, shape="chain")[0] == np.arange(-1, 19)).all()
    assert (synth.random_parents(13, 2, 20, shape="star") == -1).all()


def test_accepted_paths_are_root_to_node_chains():
    par = synth.random_parents(17, 40, 60, max_depth=6)
    path, count = synth.accepted_paths(17, par, 6)
    assert path.shape == (40, 6) and count.shape == (40,)
    for b in range(40):
        L = count[b] - 1
        assert 0 <= L <= 6
        assert (path[b, L:] == -1).all()
        nodes = path[b, :L]
        for d, v in enumerate(nodes):  # each node's parent is the previous one (the root first)
            assert par[b, v] == (nodes[d - 1] if d else -1)
            assert v >= d
