"""The allocation-free chain entry point (spec_verify_chain_noalloc).

Callers that cannot give the library a workspace (an engine that owns every device
allocation, a plugin interface that passes only input and output buffers) use this
entry point; it takes its scratch from a fixed array inside the library.  Here it is
called through the C ABI, twice in a row on each input, and its outputs must agree
with those of spec_verify_chain given a workspace within the parity rule the other
GPU tests use: identical tokens and counts, except on rows where the fp64 oracle
saw a decision within 1e-5 of its boundary (the two entry points may run different
kernels, whose fp32 reductions round differently).
This file is collected last so that a failure here does not stop the rest of a
`-x` run; it passes alone and after the other tests alike.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_verification_53_gb300 import synth
from _harness import MARGIN, oracle_chain

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _noalloc_call(lib, w, t, d, tok, temp, seed, offset):
    import torch
    B, K1, V = w["target"].shape
    K = K1 - 1
    ot = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ap = torch.full((B, K), -7.0, dtype=torch.float32, device="cuda")
    tdt = 1 if w["target"].dtype == np.uint16 else 0
    ddt = 1 if w["draft"].dtype == np.uint16 else 0
    vp = ctypes.c_void_p
    st = lib.spec_verify_chain_noalloc(vp(t.data_ptr()), tdt, vp(d.data_ptr()), ddt, w["draft_kind"],
                                       vp(tok.data_ptr()), vp(temp.data_ptr()), B, K, V, seed, offset,
                                       vp(ot.data_ptr()), vp(oc.data_ptr()), vp(ap.data_ptr()),
                                       vp(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0, st
    return ot.cpu().numpy(), oc.cpu().numpy(), ap.cpu().numpy()


@pytest.mark.parametrize("case", ["single_stream", "mixed", "tiny_fp32", "moderate"])
def test_noalloc_matches_workspace_entry_point(case):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    from speculative_decoding_verification_53_gb300 import build
    build.build()
    lib = sv.lib()
    if case == "single_stream":
        w = synth.single_stream(seed=31, B=2)
    elif case == "mixed":
        w = synth.mixed_batch(seed=32, B=3, K=5, V=32000)
    elif case == "moderate":  # a batch the automatic kernel choice walks (no scratch used)
        w = synth.mixed_batch(seed=34, B=128, K=5, V=32000)
    else:
        w = synth.tiny_chain(seed=33, V=1024, K=4, B=1)
    t, d, tok, temp = _dev(w["target"]), _dev(w["draft"]), _dev(w["tokens"]), _dev(w["temperature"])
    B, K1, V = w["target"].shape
    kind = "probs" if w["draft_kind"] == 0 else "logits"
    ws = torch.zeros(sv.spec_verify_workspace_size(B, K1 - 1, V), dtype=torch.uint8, device="cuda")
    for call, (seed, offset) in enumerate([(5, 0), (5, 1)]):  # two calls in a row
        rt, rc, ra = sv.spec_verify_chain(t, d, tok, temp, seed, offset, draft_kind=kind, workspace=ws,
                                          want_accept_prob=True)
        torch.cuda.synchronize()
        nt, nc, na = _noalloc_call(lib, w, t, d, tok, temp, seed, offset)
        rt, rc, ra = rt.cpu().numpy(), rc.cpu().numpy(), ra.cpu().numpy()
        o = oracle_chain(w, seed=seed, offset=offset)
        same = (nt == rt).all(1) & (nc == rc)
        assert all(o["margin"][i] < MARGIN for i in np.nonzero(~same)[0]), (call, nt, rt)
        np.testing.assert_allclose(na[same], ra[same], rtol=0, atol=1e-5)
        assert (nc >= 1).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import speculative_decoding_verification_53_gb300 as sv
    lib = sv.lib()
    vp = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    B, K, V = 65535, 64, 152064
    assert sv.spec_verify_workspace_size(B, K, V) > (256 << 10)
    st = lib.spec_verify_chain_noalloc(vp, 1, vp, 1, 1, vp, vp, B, K, V, 0, 0, vp, vp, None, None)
    assert st == sv.SV_ERR_UNSUPPORTED


def test_noalloc_scratch_limit_edges():
    """B = 32768 rows need exactly the 256 KiB of scratch and run (matching the
    workspace entry point); one row more is refused before anything is launched."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    lib = sv.lib()
    B, K, V = 32768, 1, 16
    assert sv.spec_verify_workspace_size(B, K, V) == (256 << 10)
    assert sv.spec_verify_workspace_size(B + 1, K, V) > (256 << 10)
    w = synth.tiny_chain(seed=35, V=V, K=K, B=B)
    t, d, tok, temp = _dev(w["target"]), _dev(w["draft"]), _dev(w["tokens"]), _dev(w["temperature"])
    ws = torch.zeros(sv.spec_verify_workspace_size(B, K, V), dtype=torch.uint8, device="cuda")
    for offset in (0, 1):
        rt, rc, _ = sv.spec_verify_chain(t, d, tok, temp, 3, offset, draft_kind="logits", workspace=ws)
        torch.cuda.synchronize()
        nt, nc, _ = _noalloc_call(lib, w, t, d, tok, temp, 3, offset)
        rt, rc = rt.cpu().numpy(), rc.cpu().numpy()
        same = (nt == rt).all(1) & (nc == rc)
        if not same.all():
            rows = np.nonzero(~same)[0]
            o = oracle_chain(w, seed=3, offset=offset, rows=rows)
            assert (o["margin"] < MARGIN).all(), rows[:8]
        assert (nc >= 1).all()
    vp = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    st = lib.spec_verify_chain_noalloc(vp, 0, vp, 0, 1, vp, vp, B + 1, K, V, 0, 0, vp, vp, None, None)
    assert st == sv.SV_ERR_UNSUPPORTED
