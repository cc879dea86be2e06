"""Each kernel family (all-positions staged, position-parallel, shared-memory staged walk,
register streaming, ring-streamed walk) against the oracle on the same aligned inputs;
the family is forced through the SPEC_VERIFY_PATH environment variable in a child
process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("path", ["eager", "spec", "staged", "stream", "ring"])
def test_kernel_family_matches_oracle(path):
    env = dict(os.environ, SPEC_VERIFY_PATH=path)
    res = subprocess.run([sys.executable, os.path.join(HERE, "_path_check.py")], env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert res.stdout.strip().startswith("ok")


def test_explicit_small_workspace_falls_back():
    import numpy as np
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    from speculative_decoding_verification_53_gb300 import synth
    from _harness import compare, oracle_chain, to_dev
    w = synth.single_stream(seed=1, B=1)
    tiny = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for ws in (tiny, None):
        ot, oc, _ = sv.spec_verify_chain(to_dev(w["target"]), to_dev(w["draft"]), to_dev(w["tokens"]),
                                         to_dev(w["temperature"]), 0, 0, draft_kind="probs", workspace=ws)
        g = dict(tokens=ot.cpu().numpy(), count=oc.cpu().numpy())
        assert compare(g, oracle_chain(w, seed=0, offset=0)) <= 1
    need = sv.spec_verify_workspace_size(1, 5, 128256)
    assert need > 0
    full = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(3):  # the workspace is left zeroed after every call and can be reused
        ot, oc, _ = sv.spec_verify_chain(to_dev(w["target"]), to_dev(w["draft"]), to_dev(w["tokens"]),
                                         to_dev(w["temperature"]), 0, 0, draft_kind="probs", workspace=full)
        assert compare(dict(tokens=ot.cpu().numpy(), count=oc.cpu().numpy()), oracle_chain(w, seed=0, offset=0)) <= 1
    torch.cuda.synchronize()
    assert int(full[:4].view(torch.int32).item()) == 0
