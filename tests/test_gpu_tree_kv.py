"""GPU parity of the tree-attention mask and the accepted-path KV compaction.

Both are integer / byte work, so the bar is bit-exact equality with the oracle on
the same seeded inputs: every mask word, depth and valid flag; every byte of every
cache buffer after the compaction (moved rows and untouched ones alike).
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_53_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_53_gb300 import build
    build.build()
    import speculative_decoding_verification_53_gb300 as m
    m.lib()
    return m


def _gpu_mask(sv, par):
    import torch
    m, d, v = sv.spec_tree_mask(torch.from_numpy(np.ascontiguousarray(par, np.int32)).cuda())
    torch.cuda.synchronize()
    return m.cpu().numpy().view(np.uint32), d.cpu().numpy(), v.cpu().numpy()


@pytest.mark.parametrize("shape", ["bfs", "random", "chain", "star"])
@pytest.mark.parametrize("N", [1, 31, 32, 33, 60, 97, 255, 512, 1024])
def test_mask_matches_oracle(sv, shape, N):
    par = synth.random_parents(21, 4, N, shape=shape, max_depth=8 if N < 256 else 24)
    m, d, v = _gpu_mask(sv, par)
    o = oracle.tree_mask(par)
    assert (m == o["mask"]).all()
    assert (d == o["depth"]).all()
    assert (v == o["valid"]).all() and (v == 1).all()


@pytest.mark.parametrize("B,N", [(2048, 60), (300, 200)])
def test_mask_invalid_rows_and_many_rows(sv, B, N):
    par = synth.random_parents(22, B, N)
    rng = np.random.default_rng(3)
    bad = rng.choice(B, 40, replace=False)  # four kinds of malformed parent entry
    for k, b in enumerate(bad):
        i = int(rng.integers(0, N))
        par[b, i] = [i, i + 5 if i + 5 < N else i, -2, 1 << 20][k % 4]
    m, d, v = _gpu_mask(sv, par)
    o = oracle.tree_mask(par)
    assert (v == o["valid"]).all() and (v == 0).sum() >= 30
    assert (m == o["mask"]).all() and (d == o["depth"]).all()


def test_mask_bad_arguments_and_empty_batch(sv):
    import ctypes
    lib = sv.lib()
    vp = ctypes.c_void_p(16)
    assert lib.spec_tree_mask(vp, 1, 0, vp, None, None, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_tree_mask(vp, 1, 1025, vp, None, None, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_tree_mask(None, 1, 8, vp, None, None, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_tree_mask(None, 0, 8, None, None, None, None) == sv.SV_OK


def _oracle_kv(bufs, path, count, base):
    """Oracle compaction of [B][H][R][row_bytes] byte buffers: (b, h) pairs are batch rows."""
    out = []
    for buf in bufs:
        B, H, R, rb = buf.shape
        flat = buf.reshape(B * H, R, rb)
        res = oracle.kv_compact(flat, np.repeat(path, H, axis=0), np.repeat(count, H), np.repeat(base, H))
        out.append(res.reshape(B, H, R, rb))
    return out


def _kv_case(seed, B, N, D, H, R, width, n_buf):
    par = synth.random_parents(seed, B, N, max_depth=D)
    path, count = synth.accepted_paths(seed, par, D)
    base = np.random.default_rng([seed, 5]).integers(0, R - N + 1, B).astype(np.int32)
    kv = synth.kv_cache(seed, n_buf, B, H, R, width)
    return kv, path, count, base


@pytest.mark.parametrize("width,dtype", [(256, "bf16"), (12, "u8"), (6, "u8"), (64, "u8")])
def test_kv_compact_matches_oracle(sv, width, dtype):
    import torch
    B, N, D, H, R, n_buf = 12, 40, 6, 3, 64, 5
    kv, path, count, base = _kv_case(31, B, N, D, H, R, width, n_buf)
    count[0] = 0            # an invalid verify row
    path[1, 1] = 0; count[1] = max(count[1], 3)  # path[1] < 1: invalid
    if dtype == "bf16":
        dev = [torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16) for k in kv]
        dev = [t.view(B, H, R, width // 2) for t in dev]
    else:
        dev = [torch.from_numpy(k).cuda() for k in kv]
    sv.spec_kv_compact(dev, torch.from_numpy(path).cuda(), torch.from_numpy(count).cuda(),
                       torch.from_numpy(base).cuda())
    torch.cuda.synchronize()
    want = _oracle_kv(list(kv), path, count, base)
    for t, w in zip(dev, want):
        got = t.view(torch.uint8).cpu().numpy().reshape(w.shape) if dtype == "bf16" else t.cpu().numpy()
        assert (got == w).all()


def test_kv_compact_permuted_layout_and_no_base(sv):
    """A [B][rows][heads][dim] cache passed as a permuted [B][heads][rows][dim] view."""
    import torch
    B, N, D, H, R, dim = 6, 30, 5, 4, 40, 32
    par = synth.random_parents(41, B, N, max_depth=D)
    path, count = synth.accepted_paths(41, par, D)
    raw = [np.random.default_rng([41, k]).integers(0, 256, (B, R, H, dim * 2), dtype=np.uint8) for k in range(3)]
    dev = [torch.from_numpy(r).cuda() for r in raw]
    views = [t.view(torch.bfloat16).permute(0, 2, 1, 3) for t in dev]
    sv.spec_kv_compact(views, torch.from_numpy(path).cuda(), torch.from_numpy(count).cuda(), None)
    torch.cuda.synchronize()
    want = _oracle_kv([np.ascontiguousarray(r.transpose(0, 2, 1, 3)) for r in raw], path, count,
                      np.zeros(B, np.int32))
    for t, w in zip(dev, want):
        assert (t.cpu().numpy().transpose(0, 2, 1, 3) == w).all()


def test_kv_compact_max_depth_and_long_paths(sv):
    import torch
    B, N, D, H, R, width = 4, 200, 64, 2, 260, 16
    par = synth.random_parents(51, B, N, shape="chain")
    path = np.full((B, D), -1, np.int32)
    count = np.zeros(B, np.int32)
    rng = np.random.default_rng(9)
    for b in range(B):  # increasing paths of length up to 64 with gaps
        L = [64, 40, 9, 1][b]
        path[b, :L] = np.sort(rng.choice(np.arange(N), L, replace=False))
        count[b] = L + 1
    kv = synth.kv_cache(51, 2, B, H, R, width)
    dev = [torch.from_numpy(k).cuda() for k in kv]
    base = np.array([0, 3, 60, 259], np.int32)
    sv.spec_kv_compact(dev, torch.from_numpy(path).cuda(), torch.from_numpy(count).cuda(),
                       torch.from_numpy(base).cuda())
    torch.cuda.synchronize()
    want = _oracle_kv(list(kv), path, count, base)
    for t, w in zip(dev, want):
        assert (t.cpu().numpy() == w).all()
    assert par.shape == (B, N)


def test_kv_compact_after_gpu_tree_verify(sv):
    """Tree verify then compaction on the GPU: the leading cache rows spell the accepted tokens."""
    import torch
    from _harness import to_dev, oracle_tree, MARGIN
    w = synth.tree(seed=61, temperature=1.0, B=8, N=30, V=2048, max_depth=6)
    d = {k: to_dev(w[k]) for k in ("target", "draft", "node_tokens", "parent", "temperature")}
    toks, cnt, pth = sv.spec_verify_tree(d["target"], d["draft"], d["node_tokens"], d["parent"], d["temperature"],
                                         w["max_depth"], w["seed"], w["offset"], draft_kind="logits")
    B, N = w["node_tokens"].shape
    kv = torch.zeros((B, 1, 2 + N, 4), dtype=torch.uint8, device="cuda")
    tok_bytes = torch.from_numpy((w["node_tokens"][:, :, None] >> np.arange(0, 32, 8)) & 0xFF).to(torch.uint8)
    kv[:, 0, 2:2 + N, :] = tok_bytes.cuda()
    base = torch.full((B,), 2, dtype=torch.int32, device="cuda")
    sv.spec_kv_compact([kv], pth, cnt, base)
    torch.cuda.synchronize()
    kv, toks, cnt = kv.cpu().numpy(), toks.cpu().numpy(), cnt.cpu().numpy()
    o = oracle_tree(w)
    for b in range(B):
        L = cnt[b] - 1
        got = kv[b, 0, 2:2 + L].astype(np.int64) @ (1 << np.arange(0, 32, 8))
        assert got.tolist() == toks[b, :L].tolist()
        if not (toks[b] == o["tokens"][b]).all():
            assert o["margin"][b] < MARGIN


def test_kv_compact_bad_arguments(sv):
    import ctypes
    lib = sv.lib()
    vp = ctypes.c_void_p(16)
    arr = (ctypes.c_void_p * 1)(16)
    f = lib.spec_kv_compact
    assert f(arr, 0, 0, 0, 1, 16, 16, 8, vp, vp, None, 1, 4, None) == sv.SV_ERR_INVALID_ARG   # no buffers
    assert f(arr, 1, 0, 0, 1, 8, 16, 8, vp, vp, None, 1, 4, None) == sv.SV_ERR_INVALID_ARG    # row > stride
    assert f(arr, 1, 0, 0, 1, 16, 16, 8, vp, vp, None, 1, 65, None) == sv.SV_ERR_INVALID_ARG  # depth 65
    assert f(arr, 1, 0, 0, 1, 16, 16, 8, None, vp, None, 1, 4, None) == sv.SV_ERR_INVALID_ARG  # no path
    assert f(arr, 1, 0, 0, 1, 16, 16, 8, None, None, None, 0, 4, None) == sv.SV_OK            # empty batch


@pytest.mark.parametrize("N", [12, 70])
def test_mask_at_the_largest_batch(sv, N):
    """B = 65535 trees, the most the boundary takes, through the small-tree kernel (N <= 64)
    and the general one; one tree more is refused before anything runs."""
    import ctypes
    B = 65535
    par = synth.random_parents(23 + N, B, N, max_depth=8)
    m, d, v = _gpu_mask(sv, par)
    o = oracle.tree_mask(par)
    assert (v == o["valid"]).all() and (m == o["mask"]).all() and (d == o["depth"]).all()
    vp = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    assert sv.lib().spec_tree_mask(vp, B + 1, N, vp, None, None, None) == sv.SV_ERR_INVALID_ARG


def test_kv_compact_at_its_limits(sv):
    """256 cache tensors in one call (the most it takes) and B = 65535 batch rows, every
    byte against the oracle; 257 tensors or one row more are refused before anything runs."""
    import ctypes
    import torch
    B, N, D, H, R, width = 3, 20, 5, 2, 24, 16
    kv, path, count, base = _kv_case(51, B, N, D, H, R, width, 256)
    dev = [torch.from_numpy(k).cuda() for k in kv]
    sv.spec_kv_compact(dev, torch.from_numpy(path).cuda(), torch.from_numpy(count).cuda(),
                       torch.from_numpy(base).cuda())
    torch.cuda.synchronize()
    for t, w in zip(dev, _oracle_kv(list(kv), path, count, base)):
        assert (t.cpu().numpy() == w).all()
    B, N, D, H, R, width = 65535, 12, 4, 1, 16, 4
    kv, path, count, base = _kv_case(52, B, N, D, H, R, width, 1)
    dev = [torch.from_numpy(k).cuda() for k in kv]
    sv.spec_kv_compact(dev, torch.from_numpy(path).cuda(), torch.from_numpy(count).cuda(),
                       torch.from_numpy(base).cuda())
    torch.cuda.synchronize()
    assert (dev[0].cpu().numpy() == _oracle_kv(list(kv), path, count, base)[0]).all()
    vp = ctypes.c_void_p(16)  # never dereferenced: the size checks come first
    arr = (ctypes.c_void_p * 257)(*([16] * 257))
    f = sv.lib().spec_kv_compact
    assert f(arr, 257, 0, 0, 1, 16, 16, 8, vp, vp, None, 1, 4, None) == sv.SV_ERR_INVALID_ARG
    assert f(arr, 1, 0, 0, 1, 16, 16, 8, vp, vp, None, 65536, 4, None) == sv.SV_ERR_INVALID_ARG
