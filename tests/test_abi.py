"""The C-ABI library builds, loads and exports every symbol include/*.h declares;
host-side argument checks answer without launching anything (no GPU needed)."""
import ctypes
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^SV_API\s+[^;(]*?\b(\w+)\s*\(", text, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from speculative_decoding_verification_53_gb300 import build
    build.build()
    import speculative_decoding_verification_53_gb300 as sv
    return sv.lib()


def test_header_declares_the_boundary():
    names = _declared_symbols()
    assert {"spec_verify_chain", "spec_verify_tree", "spec_greedy_accept", "spec_verify_workspace_size",
            "spec_verify_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    path = lib._name
    for name in _declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported by {path}"


def test_only_the_c_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    exported = {e for e in exported if not e.startswith("_")}
    assert exported == _declared_symbols()


def test_status_strings(lib):
    import speculative_decoding_verification_53_gb300 as sv
    for code in range(6):
        assert sv.spec_verify_status_string(code).startswith("SV_")
    assert "unknown" in sv.spec_verify_status_string(99)


def test_argument_errors_are_reported_before_any_launch(lib):
    import speculative_decoding_verification_53_gb300 as sv
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    ch = lib.spec_verify_chain
    # negative B, K too large, V = 0, bad dtype, probs with a bf16 draft dtype
    assert ch(vp, 0, vp, 0, 0, vp, vp, -1, 4, 100, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert ch(vp, 0, vp, 0, 0, vp, vp, 1, 65, 100, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert ch(vp, 0, vp, 0, 0, vp, vp, 1, 4, 0, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert ch(vp, 7, vp, 0, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert ch(vp, 0, vp, 1, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert ch(None, 0, vp, 0, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    # an empty batch is a successful no-op
    assert ch(None, 0, None, 0, 0, None, None, 0, 4, 100, 0, 0, None, None, None, None, 0, None) == sv.SV_OK
    g = lib.spec_greedy_accept
    assert g(vp, 0, vp, 1, -1, 100, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert g(vp, 0, None, 1, 3, 100, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    t = lib.spec_verify_tree
    # N = 0, depth 0, depth 65, N over the limit, missing parent array
    assert t(vp, 0, vp, 0, 1, vp, vp, vp, 1, 0, 100, 4, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert t(vp, 0, vp, 0, 1, vp, vp, vp, 1, 8, 100, 0, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert t(vp, 0, vp, 0, 1, vp, vp, vp, 1, 8, 100, 65, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert t(vp, 0, vp, 0, 1, vp, vp, vp, 1, 1025, 100, 4, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert t(vp, 0, vp, 0, 1, vp, None, vp, 1, 8, 100, 4, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    tr = lib.spec_verify_tree_rule
    # an unknown sibling rule; draft probabilities with a bf16 draft dtype; an empty batch
    assert tr(vp, 0, vp, 0, 1, vp, vp, vp, 1, 8, 100, 4, 2, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert tr(vp, 0, vp, 1, 0, vp, vp, vp, 1, 8, 100, 4, 0, 0, 0, vp, vp, vp, None) == sv.SV_ERR_INVALID_ARG
    assert tr(None, 0, None, 0, 1, None, None, None, 0, 8, 100, 4, 1, 0, 0, None, None, None, None) == sv.SV_OK
    sa = lib.spec_sample_and_verify
    # negative B, a bad dtype, no draft logits or drafted-token output with K > 0, an empty batch
    assert sa(vp, 0, vp, 0, vp, -1, 4, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert sa(vp, 0, vp, 5, vp, 1, 4, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert sa(vp, 0, None, 0, vp, 1, 4, 100, 0, 0, vp, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert sa(vp, 0, vp, 0, vp, 1, 4, 100, 0, 0, None, vp, vp, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert sa(None, 0, None, 0, None, 0, 4, 100, 0, 0, None, None, None, None, None, 0, None) == sv.SV_OK
    na = lib.spec_verify_chain_noalloc
    # checked like spec_verify_chain before the device is touched; scratch over 256 KiB is refused
    assert na(vp, 0, vp, 0, 0, vp, vp, 1, 65, 100, 0, 0, vp, vp, None, None) == sv.SV_ERR_INVALID_ARG
    assert na(vp, 7, vp, 0, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None) == sv.SV_ERR_INVALID_ARG
    assert na(vp, 0, vp, 1, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None) == sv.SV_ERR_INVALID_ARG
    assert na(None, 0, vp, 0, 0, vp, vp, 1, 4, 100, 0, 0, vp, vp, None, None) == sv.SV_ERR_INVALID_ARG
    assert na(vp, 0, vp, 0, 0, vp, vp, 40000, 4, 100, 0, 0, vp, vp, None, None) == sv.SV_ERR_UNSUPPORTED
    assert na(None, 0, None, 0, 0, None, None, 0, 4, 100, 0, 0, None, None, None, None) == sv.SV_OK
    ws = lib.spec_verify_workspace_size
    assert ws(-1, 4, 100) == 0 and ws(1, 65, 100) == 0 and ws(1, 4, 0) == 0
    assert ws(1, 5, 128256) == 256 and ws(1000, 5, 128256) == 8192  # one 8-byte word per row, 256-byte rounded
    c = lib.spec_verify_count_invalid
    # negative B, B over 2^24, no output, no counts with B > 0
    assert c(vp, -1, vp, None) == sv.SV_ERR_INVALID_ARG
    assert c(vp, (1 << 24) + 1, vp, None) == sv.SV_ERR_INVALID_ARG
    assert c(vp, 4, None, None) == sv.SV_ERR_INVALID_ARG
    assert c(None, 4, vp, None) == sv.SV_ERR_INVALID_ARG


def test_host_round_trip_sizes_and_argument_errors(lib):
    """spec_verify_host_sizes: the packed input's parts start on 256-byte boundaries in the
    documented order and cover their arrays; the output is tokens then counts.  The host
    entry rejects bad sizes and NULL buffers before anything is enqueued."""
    import speculative_decoding_verification_53_gb300 as sv
    off = (ctypes.c_size_t * 4)()
    nin, nout = ctypes.c_size_t(0), ctypes.c_size_t(0)
    B, K, V = 3, 5, 1001
    st = lib.spec_verify_host_sizes(B, K, V, sv.SV_BF16, sv.SV_F32, sv.SV_DRAFT_PROBS, ctypes.cast(off, ctypes.c_void_p),
                                    ctypes.byref(nin), ctypes.byref(nout))
    assert st == sv.SV_OK
    parts = [B * (K + 1) * V * 2, B * K * V * 4, B * K * 4, B * 4]  # target, draft, tokens, temperature
    assert off[0] == 0 and all(o % 256 == 0 for o in off) and nin.value % 256 == 0
    for i in range(3):
        assert off[i] + parts[i] <= off[i + 1] < off[i] + parts[i] + 256
    assert off[3] + parts[3] <= nin.value < off[3] + parts[3] + 256
    assert nout.value == B * (K + 2) * 4
    hs = lib.spec_verify_host_sizes
    nul = None
    assert hs(1, 65, 100, 0, 0, 0, nul, nul, nul) == sv.SV_ERR_INVALID_ARG           # K over 64
    assert hs(1, 4, 100, 1, 1, 0, nul, nul, nul) == sv.SV_ERR_INVALID_ARG            # bf16 probabilities
    assert hs(1, 4, 100, 2, 0, 0, nul, nul, nul) == sv.SV_ERR_INVALID_ARG            # unknown dtype
    assert hs(0, 4, 100, 0, 0, 0, nul, nul, nul) == sv.SV_OK
    h = lib.spec_verify_chain_host
    vp = ctypes.c_void_p(16)  # never dereferenced: the checks come first
    assert h(vp, vp, vp, vp, 0, 0, 0, -1, 4, 100, 0, 0, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert h(vp, None, vp, vp, 0, 0, 0, 1, 4, 100, 0, 0, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert h(vp, vp, vp, None, 0, 0, 0, 1, 4, 100, 0, 0, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert h(None, None, None, None, 0, 0, 0, 0, 4, 100, 0, 0, None, 0, None) == sv.SV_OK  # empty batch


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    import speculative_decoding_verification_53_gb300 as sv
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sv.lib()
