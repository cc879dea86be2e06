"""spec_verify_chain_host: the round trip from pinned host buffers (one packed copy in, the
verify, one copy out) gives the outputs spec_verify_chain gives on the same inputs, on
two streams used alternately, and rejects NULL buffers without touching the device."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_verification_53_gb300 import synth
from _harness import compare, oracle_chain, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["single_stream", "mixed"])
def test_host_round_trip_matches_device_entry(case):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    w = synth.single_stream(seed=41, B=2) if case == "single_stream" else synth.mixed_batch(seed=42, B=6, K=4, V=8192)
    kind = "probs" if w["draft_kind"] == 0 else "logits"
    B, K1, V = w["target"].shape
    K = K1 - 1
    tdt = torch.bfloat16 if w["target"].dtype == np.uint16 else torch.float32
    ddt = torch.bfloat16 if w["draft"].dtype == np.uint16 else torch.float32
    offs, nin, nout = sv.spec_verify_host_sizes(B, K, V, target_dtype=tdt, draft_dtype=ddt, draft_kind=kind)
    assert all(o % 256 == 0 for o in offs) and nin % 256 == 0 and nout == B * (K + 2) * 4
    hin = torch.zeros(nin, dtype=torch.uint8).pin_memory()
    hv = hin.numpy()
    for o, k in zip(offs, ("target", "draft", "tokens", "temperature")):
        a = np.ascontiguousarray(w[k])
        hv[o:o + a.nbytes] = np.frombuffer(a.tobytes(), dtype=np.uint8)
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    dins = [torch.empty(nin, dtype=torch.uint8, device="cuda") for _ in range(2)]
    douts = [torch.empty(nout, dtype=torch.uint8, device="cuda") for _ in range(2)]
    houts = [torch.zeros(nout, dtype=torch.uint8).pin_memory() for _ in range(2)]
    wss = [torch.zeros(max(sv.spec_verify_workspace_size(B, K, V), 256), dtype=torch.uint8, device="cuda")
           for _ in range(2)]
    for i in range(4):  # calls alternate between the two streams
        j = i & 1
        sv.spec_verify_chain_host(hin, dins[j], houts[j], douts[j], B, K, V, 9, i, target_dtype=tdt, draft_dtype=ddt,
                                  draft_kind=kind, workspace=wss[j], stream=streams[j])
    torch.cuda.synchronize()
    for j, i in ((0, 2), (1, 3)):  # the last call on each stream: offsets 2 and 3
        out = houts[j].view(torch.int32).numpy()
        tokens, count = out[:B * (K + 1)].reshape(B, K + 1), out[B * (K + 1):]
        rt, rc, _ = sv.spec_verify_chain(to_dev(w["target"]), to_dev(w["draft"]), to_dev(w["tokens"]),
                                         to_dev(w["temperature"]), 9, i, draft_kind=kind)
        assert np.array_equal(tokens, rt.cpu().numpy()) and np.array_equal(count, rc.cpu().numpy())
        assert compare(dict(tokens=tokens, count=count), oracle_chain(w, seed=9, offset=i)) <= 1


def test_host_entry_rejects_null_buffers():
    import speculative_decoding_verification_53_gb300 as sv
    lib = sv.lib()
    vp = ctypes.c_void_p(16)  # never dereferenced: the argument check comes first
    st = lib.spec_verify_chain_host(None, vp, vp, vp, 1, 0, 0, 1, 5, 1000, 0, 0, None, 0, None)
    assert st == sv.SV_ERR_INVALID_ARG
    st = lib.spec_verify_chain_host(vp, vp, vp, vp, 1, 0, 0, 1, 65, 1000, 0, 0, None, 0, None)  # K beyond 64
    assert st == sv.SV_ERR_INVALID_ARG
