"""Pins of the oracle's tree-attention mask and accepted-path KV compaction (no GPU).

The mask is tied to networkx (ancestor sets and root distances of the same tree
as a graph) and to closed forms (a chain gives the lower triangle, a star the
identity).  The compaction is tied to the gather identity it must equal when
every source lies at or after its destination, to rows it must not touch, and
end to end to the tree verify: after compacting a cache whose rows hold the
node tokens, the leading rows must spell the accepted tokens.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth

nx = pytest.importorskip("networkx")


def _bits(mask_row, N):
    return [j for j in range(N) if (int(mask_row[j // 32]) >> (j % 32)) & 1]


@pytest.mark.parametrize("shape", ["bfs", "random", "chain", "star"])
@pytest.mark.parametrize("N", [1, 31, 32, 33, 60, 97])
def test_mask_equals_networkx_ancestors(shape, N):
    par = synth.random_parents(5, 3, N, shape=shape)
    o = oracle.tree_mask(par)
    assert (o["valid"] == 1).all()
    for b in range(3):
        g = nx.DiGraph()
        g.add_node("root")
        for i in range(N):
            g.add_edge("root" if par[b, i] < 0 else int(par[b, i]), i)
        dist = nx.single_source_shortest_path_length(g, "root")
        for i in range(N):
            want = sorted([a for a in nx.ancestors(g, i) if a != "root"] + [i])
            assert _bits(o["mask"][b, i], N) == want
            assert o["depth"][b, i] == dist[i]


def test_mask_closed_forms_and_padding_bits():
    N = 70
    chain = oracle.tree_mask(synth.random_parents(0, 1, N, shape="chain"))
    star = oracle.tree_mask(synth.random_parents(0, 1, N, shape="star"))
    dense_chain = np.unpackbits(chain["mask"][0].view(np.uint8), bitorder="little").reshape(N, -1)[:, :N]
    dense_star = np.unpackbits(star["mask"][0].view(np.uint8), bitorder="little").reshape(N, -1)[:, :N]
    assert (dense_chain == np.tril(np.ones((N, N), np.uint8))).all()
    assert (dense_star == np.eye(N, dtype=np.uint8)).all()
    assert (chain["depth"][0] == np.arange(1, N + 1)).all() and (star["depth"][0] == 1).all()
    # bits at or above N in the last word stay clear
    assert (chain["mask"][0, :, -1] >> np.uint32(N % 32) == 0).all()


def test_mask_malformed_rows_are_invalid_and_zero():
    par = synth.random_parents(3, 4, 40)
    par[1, 7] = 7            # self parent
    par[2, 9] = 12           # parent after the child
    par[3, 0] = -2           # below -1
    o = oracle.tree_mask(par)
    assert list(o["valid"]) == [1, 0, 0, 0]
    assert (o["mask"][1:] == 0).all() and (o["depth"][1:] == 0).all()


def _kv_case(seed, B, N, D, rows, rb):
    par = synth.random_parents(seed, B, N)
    path, count = synth.accepted_paths(seed, par, D)
    base = np.random.default_rng(seed).integers(0, rows - N + 1, B).astype(np.int32)
    kv = np.random.default_rng([seed, 1]).integers(0, 256, (B, rows, rb), dtype=np.uint8)
    return kv, path, count, base


@pytest.mark.parametrize("seed", range(6))
def test_kv_compact_is_the_gather_of_the_original_rows(seed):
    kv, path, count, base = _kv_case(seed, 8, 60, 6, 80, 24)
    out = oracle.kv_compact(kv, path, count, base)
    for b in range(8):
        L = count[b] - 1
        dst = base[b] + np.arange(L)
        src = base[b] + path[b, :L]
        assert (out[b, dst] == kv[b, src]).all()                  # gather from the ORIGINAL cache
        keep = np.setdiff1d(np.arange(kv.shape[1]), dst)
        assert (out[b, keep] == kv[b, keep]).all()                # everything else untouched


def test_kv_compact_overlapping_shift_reads_before_it_writes():
    kv = np.arange(8, dtype=np.uint8).reshape(1, 8, 1)
    out = oracle.kv_compact(kv, np.array([[1, 2, 3]], np.int32), np.array([4], np.int32), np.array([0], np.int32))
    assert out[0, :, 0].tolist() == [1, 2, 3, 3, 4, 5, 6, 7]


def test_kv_compact_identity_and_invalid_rows_are_untouched():
    kv, path, count, base = _kv_case(9, 5, 30, 6, 40, 8)
    path[0, :3] = [0, 1, 2]; count[0] = 4                         # already in place
    count[1] = 0                                                  # invalid verify row
    path[2, :2] = [3, 0]; count[2] = 3                            # path[1] < 1
    base[3] = 40 - 1; path[3, :1] = [5]; count[3] = 2             # source past the end
    count[4] = 8                                                  # longer than max_depth
    out = oracle.kv_compact(kv, path, count, base)
    assert (out == kv).all()


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_kv_compact_after_tree_verify_spells_the_accepted_tokens(T):
    """Cache row base+i holds node i's token; after the verify and the compaction the
    first count-1 rows hold the emitted tokens but the last, in order."""
    w = synth.tree(seed=4, temperature=T, B=6, N=24, V=512, max_depth=5)
    o = oracle.verify_tree(w["target"], w["draft"], w["node_tokens"], w["parent"], w["temperature"],
                           w["max_depth"], w["seed"], w["offset"], draft_kind=w["draft_kind"])
    B, N = w["node_tokens"].shape
    base = np.full(B, 3, np.int32)
    kv = np.zeros((B, 3 + N + 2, 4), np.uint8)
    kv[:, 3:3 + N, :] = (w["node_tokens"][:, :, None] >> np.arange(0, 32, 8)) & 0xFF
    out = oracle.kv_compact(kv, o["path"], o["count"], base)
    for b in range(B):
        L = o["count"][b] - 1
        got = out[b, 3:3 + L].astype(np.int64) @ (1 << np.arange(0, 32, 8))
        assert got.tolist() == o["tokens"][b, :L].tolist()
