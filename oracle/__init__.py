"""Oracle for the speculative-decoding verify/accept step -- TEST INFRASTRUCTURE.

A plain fp64, single-threaded CPU restatement (``oracle.c``) of the rule the
pages define, with a ctypes wrapper over numpy arrays.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg use
it; the product library never imports it and shares no code with it.

Sources: "[논문 리뷰] Fast Inference from Transformers via Speculative
Decoding", section 2 (accept with min(1, p/q), residual max(0, p-q), bonus
token); "Speculative Decoding and EAGLE", section "정확성 규칙" (r < p/q, the
residual, the greedy case); "Progressive Tree Drafting", section "검증"
(greedy and sampling tree acceptance).

Array conventions: logits are numpy ``float32`` (fp32) or ``uint16`` holding
bfloat16 bit patterns; draft probabilities are ``float32``.

Pins (tests/test_oracle_pins.py, test_oracle_mask_kv.py, test_oracle_sample.py):
every function is checked against something other than itself -- numpy's Philox,
closed forms, numpy argmax / searchsorted, exact law enumeration, the printed
expected-token value, brute-force tree paths, networkx ancestor sets, a gather
from the unmodified cache.  Parity unpinned: tree sampling on trees whose children
are a parent's top draft tokens (a deterministic choice, not a draw from q) has no
law to compare with; there ``verify_tree`` is checked only through the cases above
(trees drawn without replacement or i.i.d., chains as trees, greedy trees).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
DRAFT_PROBS, DRAFT_LOGITS = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, no FMA contraction,
    so x86_64 and aarch64 hosts compute identical doubles)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
                        "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32p, f32p, f64p, u64p = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_uint64))
        ci, u64 = ctypes.c_int, ctypes.c_uint64
        lib.oracle_philox4x64_10.argtypes = [u64p, u64p, u64p]
        lib.oracle_philox4x64_10.restype = None
        lib.oracle_verify_chain_u.argtypes = [vp, ci, vp, ci, ci, i32p, f32p, ci, ci, ci,
                                              f64p, f64p, i32p, i32p, f32p, f64p]
        lib.oracle_verify_chain.argtypes = [vp, ci, vp, ci, ci, i32p, f32p, ci, ci, ci,
                                            u64, u64, i32p, i32p, i32p, f32p, f64p]
        lib.oracle_greedy_accept.argtypes = [vp, ci, i32p, ci, ci, ci, i32p, i32p]
        lib.oracle_verify_tree_u.argtypes = [vp, ci, vp, ci, ci, i32p, i32p, f32p, ci, ci, ci, ci,
                                             f64p, f64p, i32p, i32p, i32p, f64p]
        lib.oracle_verify_tree.argtypes = [vp, ci, vp, ci, ci, i32p, i32p, f32p, ci, ci, ci, ci,
                                           u64, u64, i32p, i32p, i32p, i32p, f64p]
        lib.oracle_verify_tree_rule_u.argtypes = [vp, ci, vp, ci, ci, i32p, i32p, f32p, ci, ci, ci, ci, ci,
                                                  f64p, f64p, i32p, i32p, i32p, f64p]
        lib.oracle_verify_tree_rule.argtypes = [vp, ci, vp, ci, ci, i32p, i32p, f32p, ci, ci, ci, ci, ci,
                                                u64, u64, i32p, i32p, i32p, i32p, f64p]
        lib.oracle_sample_and_verify.argtypes = [vp, ci, vp, ci, f32p, ci, ci, ci, u64, u64, i32p, i32p, i32p,
                                                 i32p, f32p, f64p]
        lib.oracle_tree_mask.argtypes = [i32p, ci, ci, vp, i32p, i32p]
        lib.oracle_kv_compact.argtypes = [vp, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t, i32p, i32p, i32p,
                                          ci, ci, ci]
        for name in ("oracle_verify_chain_u", "oracle_verify_chain", "oracle_greedy_accept",
                     "oracle_verify_tree_u", "oracle_verify_tree", "oracle_tree_mask", "oracle_kv_compact",
                     "oracle_verify_tree_rule_u", "oracle_verify_tree_rule", "oracle_sample_and_verify"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def _logits_dtype(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def philox4x64_10(counter, key) -> np.ndarray:
    """One Philox4x64-10 block for a 4-word counter and a 2-word key."""
    lib = _load()
    c = _c(np.asarray(counter, dtype=np.uint64), np.uint64)
    k = _c(np.asarray(key, dtype=np.uint64), np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    lib.oracle_philox4x64_10(_ptr(c, ctypes.c_uint64), _ptr(k, ctypes.c_uint64),
                             _ptr(out, ctypes.c_uint64))
    return out


def _draft_args(draft, draft_kind):
    if draft is None:
        return None, F32
    if draft_kind == DRAFT_PROBS:
        if draft.dtype != np.float32:
            raise TypeError("draft probabilities must be float32")
        return draft, F32
    return draft, _logits_dtype(draft)


def verify_chain(target, draft, draft_tokens, temperature, seed, offset,
                 draft_kind=DRAFT_LOGITS, row_id=None, uniforms=None):
    """Chain verify.  target [B][K+1][V], draft [B][K][V], draft_tokens [B][K],
    temperature [B].  ``uniforms=(r, u)`` ([B][K], [B][K+1] float64) replaces the
    Philox stream.  Returns dict(tokens, count, accept_prob, margin, n_invalid)."""
    lib = _load()
    target = np.ascontiguousarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    tdt = _logits_dtype(target)
    draft = None if draft is None else np.ascontiguousarray(draft)
    draft, ddt = _draft_args(draft, draft_kind)
    if draft is not None and draft.shape != (B, K, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, K, V)}")
    toks = _c(draft_tokens, np.int32).reshape(B, K)
    temps = _c(temperature, np.float32).reshape(B)
    out_t = np.full((B, K + 1), -1, np.int32)
    out_c = np.zeros(B, np.int32)
    out_ap = np.full((B, max(K, 1)), -1, np.float32)
    out_m = np.zeros(B, np.float64)
    dptr = None if draft is None else draft.ctypes.data
    if uniforms is None:
        rid = None if row_id is None else _c(row_id, np.int32)
        n = lib.oracle_verify_chain(target.ctypes.data, tdt, dptr, ddt, draft_kind,
                                    _ptr(toks, ctypes.c_int32), _ptr(temps, ctypes.c_float), B, K, V,
                                    ctypes.c_uint64(seed), ctypes.c_uint64(offset),
                                    _ptr(rid, ctypes.c_int32), _ptr(out_t, ctypes.c_int32),
                                    _ptr(out_c, ctypes.c_int32), _ptr(out_ap, ctypes.c_float),
                                    _ptr(out_m, ctypes.c_double))
    else:
        r = _c(uniforms[0], np.float64).reshape(B, K) if K > 0 else np.zeros((B, 1))
        u = _c(uniforms[1], np.float64).reshape(B, K + 1)
        n = lib.oracle_verify_chain_u(target.ctypes.data, tdt, dptr, ddt, draft_kind,
                                      _ptr(toks, ctypes.c_int32), _ptr(temps, ctypes.c_float), B, K, V,
                                      _ptr(r, ctypes.c_double), _ptr(u, ctypes.c_double),
                                      _ptr(out_t, ctypes.c_int32), _ptr(out_c, ctypes.c_int32),
                                      _ptr(out_ap, ctypes.c_float), _ptr(out_m, ctypes.c_double))
    return dict(tokens=out_t, count=out_c, accept_prob=out_ap[:, :K], margin=out_m, n_invalid=n)


def greedy_accept(target, draft_tokens):
    """Greedy acceptance (argmax rule) for every row.  Returns dict(tokens, count)."""
    lib = _load()
    target = np.ascontiguousarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    toks = _c(draft_tokens, np.int32).reshape(B, K)
    out_t = np.full((B, K + 1), -1, np.int32)
    out_c = np.zeros(B, np.int32)
    n = lib.oracle_greedy_accept(target.ctypes.data, _logits_dtype(target), _ptr(toks, ctypes.c_int32),
                                 B, K, V, _ptr(out_t, ctypes.c_int32), _ptr(out_c, ctypes.c_int32))
    return dict(tokens=out_t, count=out_c, n_invalid=n)


SIBLINGS_WOR, SIBLINGS_IID = 0, 1


def verify_tree(target, draft, node_tokens, parent, temperature, max_depth, seed, offset,
                draft_kind=DRAFT_LOGITS, row_id=None, uniforms=None, sibling_rule=SIBLINGS_WOR):
    """Tree verify.  target/draft [B][N+1][V] (row 0 = root, row i+1 = after node i),
    node_tokens/parent [B][N].  ``uniforms=(r, u)`` ([B][N], [B][N+1]) replaces the
    Philox stream.  sibling_rule: SIBLINGS_WOR (siblings drafted without replacement:
    a rejected token's q is zeroed and q renormalised) or SIBLINGS_IID (drafted
    i.i.d.: q unchanged).  Returns dict(tokens, count, path, margin, n_invalid)."""
    lib = _load()
    target = np.ascontiguousarray(target)
    B, N1, V = target.shape
    N = N1 - 1
    tdt = _logits_dtype(target)
    draft = None if draft is None else np.ascontiguousarray(draft)
    draft, ddt = _draft_args(draft, draft_kind)
    if draft is not None and draft.shape != (B, N + 1, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, N + 1, V)}")
    toks = _c(node_tokens, np.int32).reshape(B, N)
    par = _c(parent, np.int32).reshape(B, N)
    temps = _c(temperature, np.float32).reshape(B)
    D = int(max_depth)
    out_t = np.full((B, D + 1), -1, np.int32)
    out_c = np.zeros(B, np.int32)
    out_p = np.full((B, max(D, 1)), -1, np.int32)
    out_m = np.zeros(B, np.float64)
    dptr = None if draft is None else draft.ctypes.data
    if uniforms is None:
        rid = None if row_id is None else _c(row_id, np.int32)
        n = lib.oracle_verify_tree_rule(target.ctypes.data, tdt, dptr, ddt, draft_kind,
                                   _ptr(toks, ctypes.c_int32), _ptr(par, ctypes.c_int32),
                                   _ptr(temps, ctypes.c_float), B, N, V, D, int(sibling_rule),
                                   ctypes.c_uint64(seed), ctypes.c_uint64(offset),
                                   _ptr(rid, ctypes.c_int32), _ptr(out_t, ctypes.c_int32),
                                   _ptr(out_c, ctypes.c_int32), _ptr(out_p, ctypes.c_int32),
                                   _ptr(out_m, ctypes.c_double))
    else:
        r = _c(uniforms[0], np.float64).reshape(B, N) if N > 0 else np.zeros((B, 1))
        u = _c(uniforms[1], np.float64).reshape(B, N + 1)
        n = lib.oracle_verify_tree_rule_u(target.ctypes.data, tdt, dptr, ddt, draft_kind,
                                     _ptr(toks, ctypes.c_int32), _ptr(par, ctypes.c_int32),
                                     _ptr(temps, ctypes.c_float), B, N, V, D, int(sibling_rule),
                                     _ptr(r, ctypes.c_double), _ptr(u, ctypes.c_double),
                                     _ptr(out_t, ctypes.c_int32), _ptr(out_c, ctypes.c_int32),
                                     _ptr(out_p, ctypes.c_int32), _ptr(out_m, ctypes.c_double))
    return dict(tokens=out_t, count=out_c, path=out_p[:, :D], margin=out_m, n_invalid=n)


def sample_and_verify(target, draft, temperature, seed, offset, row_id=None):
    """Draft sampling and verify in one step: x_k ~ softmax(draft_k / T) by the Philox
    word-2 uniform of slot k (argmax for greedy rows), then the chain verify of x.
    target [B][K+1][V], draft logits [B][K][V].  Returns dict(draft_tokens, tokens,
    count, accept_prob, margin, n_invalid)."""
    lib = _load()
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, K1, V = target.shape
    K = K1 - 1
    if draft.shape != (B, K, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, K, V)}")
    temps = _c(temperature, np.float32).reshape(B)
    rid = None if row_id is None else _c(row_id, np.int32)
    xd = np.full((B, max(K, 1)), -1, np.int32)
    out_t = np.full((B, K + 1), -1, np.int32)
    out_c = np.zeros(B, np.int32)
    out_ap = np.full((B, max(K, 1)), -1, np.float32)
    out_m = np.zeros(B, np.float64)
    n = lib.oracle_sample_and_verify(target.ctypes.data, _logits_dtype(target), draft.ctypes.data,
                                     _logits_dtype(draft), _ptr(temps, ctypes.c_float), B, K, V,
                                     ctypes.c_uint64(seed), ctypes.c_uint64(offset), _ptr(rid, ctypes.c_int32),
                                     _ptr(xd, ctypes.c_int32), _ptr(out_t, ctypes.c_int32),
                                     _ptr(out_c, ctypes.c_int32), _ptr(out_ap, ctypes.c_float),
                                     _ptr(out_m, ctypes.c_double))
    return dict(draft_tokens=xd[:, :K], tokens=out_t, count=out_c, accept_prob=out_ap[:, :K], margin=out_m,
                n_invalid=n)


def tree_mask(parent):
    """Ancestor-or-self bitmask of each node: parent [B][N] -> (mask uint32 [B][N][W],
    depth int32 [B][N], valid int32 [B])."""
    lib = _load()
    par = _c(parent, np.int32)
    B, N = par.shape
    W = (N + 31) // 32
    mask = np.zeros((B, N, W), np.uint32)
    depth = np.zeros((B, N), np.int32)
    valid = np.zeros(B, np.int32)
    lib.oracle_tree_mask(_ptr(par, ctypes.c_int32), B, N, mask.ctypes.data, _ptr(depth, ctypes.c_int32),
                         _ptr(valid, ctypes.c_int32))
    return dict(mask=mask, depth=depth, valid=valid)


def kv_compact(kv, path, count, base, inplace=False):
    """Accepted-path KV compaction of kv [B][R][row_bytes] (uint8): row base+d <- row
    base+path[d] for d < count-1, in order.  Works on a copy (returned) unless
    ``inplace`` (kv must then be a C-contiguous uint8 array; it is returned)."""
    lib = _load()
    if inplace:
        if kv.dtype != np.uint8 or not kv.flags["C_CONTIGUOUS"]:
            raise ValueError("in-place compaction needs a C-contiguous uint8 array")
        out = kv
    else:
        out = np.array(kv, dtype=np.uint8, copy=True, order="C")
    B, R, rb = out.shape
    pth = _c(path, np.int32)
    D = pth.shape[1]
    cnt = _c(count, np.int32)
    bs = _c(base, np.int32)
    lib.oracle_kv_compact(out.ctypes.data, R * rb, rb, rb, _ptr(pth, ctypes.c_int32), _ptr(cnt, ctypes.c_int32),
                          _ptr(bs, ctypes.c_int32), B, D, R)
    return out
