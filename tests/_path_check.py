"""Run a set of chain parity checks in this process (used by test_gpu_paths.py with
SPEC_VERIFY_PATH set in the environment, which the library reads once)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from speculative_decoding_verification_53_gb300 import synth  # noqa: E402
from _harness import compare, gpu_chain, gpu_tree, oracle_chain, oracle_tree  # noqa: E402


def main():
    excused = 0
    w = synth.mixed_batch(seed=11, B=6, K=5, V=32000)
    excused += compare(gpu_chain(w, seed=3), oracle_chain(w, seed=3))
    w0 = synth.single_stream(seed=2, B=6)
    for s in range(6):
        ws = {k: (v[s:s + 1] if isinstance(v, np.ndarray) else v) for k, v in w0.items()}
        excused += compare(gpu_chain(ws, seed=s, offset=s), oracle_chain(ws, seed=s, offset=s))
    w = synth.large_batch(seed=4, temperature=1.0, sigma=1.0, B=3, K=8)
    excused += compare(gpu_chain(w, seed=9), oracle_chain(w, seed=9))
    from test_gpu_parity import _bad_after_first_rejection  # noqa: E402
    w = _bad_after_first_rejection()
    g = gpu_chain(w)
    assert (g["count"] == 1).all(), g["count"]
    excused += compare(g, oracle_chain(w))
    w = synth.tiny_chain(seed=8, V=4096, K=0, B=2)
    excused += compare(gpu_chain(w), oracle_chain(w))
    w = synth.tiny_chain(seed=9, V=1024, K=64, B=1, sigma=0.1)
    excused += compare(gpu_chain(w), oracle_chain(w))
    tw = synth.tree(seed=6, B=4, N=24, V=8192, max_depth=5)
    for T in (0.0, 1.0):
        tw["temperature"] = np.full(4, T, np.float32)
        excused += compare(gpu_tree(tw, seed=2), oracle_tree(tw, seed=2), keys=("tokens", "count", "path"))
    iw = synth.redraw_children_iid(synth.tree(seed=16, B=4, N=24, V=8192, max_depth=5, sigma=2.0), seed=5)
    for rule in (oracle.SIBLINGS_IID, oracle.SIBLINGS_WOR):
        excused += compare(gpu_tree(iw, seed=7, sibling_rule=rule), oracle_tree(iw, seed=7, sibling_rule=rule),
                           keys=("tokens", "count", "path"))
    cw = synth.chain_as_tree(synth.tiny_chain(seed=7, V=2048, K=6, B=8, temperature=0.8))
    excused += compare(gpu_tree(cw, seed=4), oracle_tree(cw, seed=4), keys=("tokens", "count", "path"))
    assert excused <= 2, excused
    print("ok", excused)


if __name__ == "__main__":
    main()
