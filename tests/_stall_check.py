"""Child process of test_gpu_timeout.py: run with SPEC_VERIFY_PATH=staged,
SPEC_VERIFY_CLUSTER=1 and SPEC_VERIFY_TEST_STALL=<row> (read once by the library), so
that one batch row's first bulk copy is announced but never issued and its bounded
wait runs out.  Checks that this row reports a timeout (count -1, the call's status
SV_ERR_TIMEOUT) while every other row matches the oracle."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from speculative_decoding_verification_53_gb300 import synth  # noqa: E402
from _harness import compare, gpu_chain, oracle_chain  # noqa: E402


def main():
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    stall = int(os.environ["SPEC_VERIFY_TEST_STALL"])
    w = synth.mixed_batch(seed=21, B=6, K=4, V=8192)  # even rows greedy, odd rows sampling
    for rep in range(2):  # the context stays usable: a second call behaves the same
        g = gpu_chain(w, seed=5, offset=rep)
        assert g["count"][stall] == sv.COUNT_TIMEOUT, g["count"]
        others = np.array([b for b in range(6) if b != stall])
        assert compare(g, oracle_chain(w, seed=5, offset=rep, rows=others), rows=others) <= 1
        cnt = torch.from_numpy(g["count"]).cuda()
        st = sv.spec_verify_rows_status(cnt).cpu().numpy()
        assert st.tolist() == [sv.SV_ERR_TIMEOUT, 0, 1], st
        assert sv.rows_status(cnt) == sv.SV_ERR_TIMEOUT
        assert int(sv.spec_verify_count_invalid(cnt).item()) == 0
    # a row with bad data as well: the timeout still decides the call's status
    t = w["target"].copy()
    bad = (stall + 1) % 6
    t[bad, 0, 5] = 0x7FC0  # a bf16 NaN
    g = gpu_chain(dict(w, target=t), seed=5, offset=0)
    assert g["count"][stall] == sv.COUNT_TIMEOUT and g["count"][bad] == 0, g["count"]
    st = sv.spec_verify_rows_status(torch.from_numpy(g["count"]).cuda()).cpu().numpy()
    assert st.tolist() == [sv.SV_ERR_TIMEOUT, 1, 1], st
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
