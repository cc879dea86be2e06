"""GB300 (sm_103a) speculative-decoding verify/accept library -- Python binding.

A thin ctypes layer over ``libspecverify.so`` (C ABI: ``include/spec_verify.h``).
Each function carries the name of the C entry point it calls and only marshals
arguments: torch tensors become device pointers, the current torch stream
becomes the launch stream, outputs are allocated with torch when not given.
Every step of the verify path runs in the library's CUDA kernels; there is no
fallback -- a missing library raises.

Build the library with ``python -m speculative_decoding_verification_53_gb300.build``
(or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_TIMEOUT, SV_ERR_BAD_INPUT = range(6)
SV_F32, SV_BF16 = 0, 1
SV_DRAFT_PROBS, SV_DRAFT_LOGITS = 0, 1
SV_SIBLINGS_WITHOUT_REPLACEMENT, SV_SIBLINGS_IID = 0, 1

EXPORTS = ("spec_verify_workspace_size", "spec_verify_chain", "spec_greedy_accept", "spec_verify_tree",
           "spec_verify_status_string", "spec_verify_last_cuda_error", "spec_verify_chain_noalloc",
           "spec_tree_mask", "spec_kv_compact", "spec_verify_tree_rule", "spec_sample_and_verify",
           "spec_verify_count_invalid", "spec_verify_rows_status", "spec_verify_chain_host",
           "spec_verify_host_sizes")

# out_count value of a batch row whose kernel gave up a bounded device-side wait
COUNT_TIMEOUT = -1

_lib = None


class SpecVerifyError(RuntimeError):
    """A non-zero sv_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        detail = f" ({lib().spec_verify_last_cuda_error().decode()})" if status == SV_ERR_CUDA else ""
        super().__init__(f"{where}: {spec_verify_status_string(status)}{detail}")


def lib() -> ctypes.CDLL:
    """The loaded library with argument types set (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m speculative_decoding_verification_53_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    L.spec_verify_workspace_size.argtypes = [ci, ci, ci]
    L.spec_verify_workspace_size.restype = sz
    L.spec_verify_chain.argtypes = [vp, ci, vp, ci, ci, vp, vp, ci, ci, ci, u64, u64, vp, vp, vp, vp, sz, vp]
    L.spec_verify_chain.restype = ci
    L.spec_verify_chain_noalloc.argtypes = [vp, ci, vp, ci, ci, vp, vp, ci, ci, ci, u64, u64, vp, vp, vp, vp]
    L.spec_verify_chain_noalloc.restype = ci
    L.spec_greedy_accept.argtypes = [vp, ci, vp, ci, ci, ci, vp, vp, vp]
    L.spec_greedy_accept.restype = ci
    L.spec_verify_tree.argtypes = [vp, ci, vp, ci, ci, vp, vp, vp, ci, ci, ci, ci, u64, u64, vp, vp, vp, vp]
    L.spec_verify_tree.restype = ci
    L.spec_verify_tree_rule.argtypes = [vp, ci, vp, ci, ci, vp, vp, vp, ci, ci, ci, ci, ci, u64, u64, vp, vp, vp,
                                        vp]
    L.spec_verify_tree_rule.restype = ci
    L.spec_sample_and_verify.argtypes = [vp, ci, vp, ci, vp, ci, ci, ci, u64, u64, vp, vp, vp, vp, vp, sz, vp]
    L.spec_sample_and_verify.restype = ci
    L.spec_tree_mask.argtypes = [vp, ci, ci, vp, vp, vp, vp]
    L.spec_tree_mask.restype = ci
    i64 = ctypes.c_int64
    L.spec_kv_compact.argtypes = [ctypes.POINTER(vp), ci, i64, i64, ci, i64, i64, ci, vp, vp, vp, ci, ci, vp]
    L.spec_kv_compact.restype = ci
    L.spec_verify_status_string.argtypes = [ci]
    L.spec_verify_status_string.restype = ctypes.c_char_p
    L.spec_verify_last_cuda_error.argtypes = []
    L.spec_verify_last_cuda_error.restype = ctypes.c_char_p
    L.spec_verify_count_invalid.argtypes = [vp, ci, vp, vp]
    L.spec_verify_count_invalid.restype = ci
    L.spec_verify_rows_status.argtypes = [vp, ci, vp, vp]
    L.spec_verify_rows_status.restype = ci
    L.spec_verify_chain_host.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, u64, u64, vp, sz, vp]
    L.spec_verify_chain_host.restype = ci
    L.spec_verify_host_sizes.argtypes = [ci, ci, ci, ci, ci, ci, vp, vp, vp]
    L.spec_verify_host_sizes.restype = ci
    _lib = L
    return L


def spec_verify_status_string(status: int) -> str:
    return lib().spec_verify_status_string(int(status)).decode()


def spec_verify_workspace_size(B: int, K: int, V: int) -> int:
    return int(lib().spec_verify_workspace_size(int(B), int(K), int(V)))


# ---------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dtype_code_of(dtype) -> int:
    """The sv_dtype of a torch dtype (float32 or bfloat16)."""
    torch = _torch()
    if dtype == torch.float32:
        return SV_F32
    if dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


_workspaces = {}


def _auto_workspace(B, K, V, stream):
    """A zero-initialised workspace cached per (device, stream) and grown on demand; the
    library leaves it zeroed after every call, so it is reused as is.  Calls on one stream
    never overlap, which is what the library requires of a shared workspace."""
    torch = _torch()
    need = spec_verify_workspace_size(B, K, V)
    if need == 0:
        return None
    s = torch.cuda.current_stream() if stream is None else stream
    key = (s.device.index, s.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=s.device)
        _workspaces[key] = ws
    return ws


def _kind(draft_kind) -> int:
    if draft_kind in ("probs", SV_DRAFT_PROBS):
        return SV_DRAFT_PROBS
    if draft_kind in ("logits", SV_DRAFT_LOGITS):
        return SV_DRAFT_LOGITS
    raise ValueError("draft_kind must be 'probs' or 'logits'")


# ------------------------------------------------------------ entry points

def spec_verify_chain(target_logits, draft, draft_tokens, temperature, seed: int, offset: int, *,
                      draft_kind, out_tokens=None, out_count=None, out_accept_prob=None,
                      want_accept_prob: bool = False, workspace="auto", stream=None):
    """Chain verify.  target_logits [B][K+1][V] (fp32/bf16), draft [B][K][V] (probs fp32 or
    logits), draft_tokens int32 [B][K], temperature fp32 [B] (T <= 0: greedy row).
    workspace: "auto" (a cached zeroed buffer per stream), None (none: the kernels that need
    no scratch), or a caller-owned zero-initialised uint8 CUDA tensor.
    Returns (out_tokens int32 [B][K+1], out_count int32 [B], out_accept_prob fp32 [B][K] or None)."""
    torch = _torch()
    _dev(target_logits, "target_logits")
    B, K1, V = target_logits.shape
    K = K1 - 1
    dk = _kind(draft_kind)
    _dev(draft, "draft")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    _dev(temperature, "temperature", torch.float32)
    ddt = SV_F32 if draft is None else _dtype_code(draft)
    if draft is not None and tuple(draft.shape) != (B, K, V):
        raise ValueError(f"draft shape {tuple(draft.shape)} != {(B, K, V)}")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_accept_prob is None and want_accept_prob:
        out_accept_prob = torch.empty((B, K), dtype=torch.float32, device=dev)
    if isinstance(workspace, str):
        workspace = _auto_workspace(B, K, V, stream) if B > 0 else None
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    st = lib().spec_verify_chain(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, dk,
                                 _ptr(draft_tokens), _ptr(temperature), B, K, V, int(seed), int(offset),
                                 _ptr(out_tokens), _ptr(out_count), _ptr(out_accept_prob), ws_ptr, ws_bytes,
                                 _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_chain")
    return out_tokens, out_count, out_accept_prob


def spec_verify_chain_noalloc(target_logits, draft, draft_tokens, temperature, seed: int, offset: int, *,
                              draft_kind, out_tokens=None, out_count=None, out_accept_prob=None,
                              want_accept_prob: bool = False, stream=None):
    """spec_verify_chain for callers that cannot provide a workspace: the library uses a
    fixed 256 KiB scratch array of its own (first call on a device sets it up, so make it
    before any graph capture; overlapping calls race).  Same arguments and results."""
    torch = _torch()
    _dev(target_logits, "target_logits")
    B, K1, V = target_logits.shape
    K = K1 - 1
    dk = _kind(draft_kind)
    _dev(draft, "draft")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    _dev(temperature, "temperature", torch.float32)
    ddt = SV_F32 if draft is None else _dtype_code(draft)
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_accept_prob is None and want_accept_prob:
        out_accept_prob = torch.empty((B, K), dtype=torch.float32, device=dev)
    st = lib().spec_verify_chain_noalloc(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, dk,
                                         _ptr(draft_tokens), _ptr(temperature), B, K, V, int(seed), int(offset),
                                         _ptr(out_tokens), _ptr(out_count), _ptr(out_accept_prob), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_chain_noalloc")
    return out_tokens, out_count, out_accept_prob


def spec_sample_and_verify(target_logits, draft_logits, temperature, seed: int, offset: int, *,
                           out_draft_tokens=None, out_tokens=None, out_count=None, out_accept_prob=None,
                           want_accept_prob: bool = False, workspace="auto", stream=None):
    """Draft sampling and verify in one call: x_k ~ softmax(draft_logits_k / T) (argmax for
    greedy rows), then the chain verify of those tokens.  target_logits [B][K+1][V],
    draft_logits [B][K][V], temperature fp32 [B].  Returns (out_draft_tokens [B][K],
    out_tokens [B][K+1], out_count [B], out_accept_prob [B][K] or None)."""
    torch = _torch()
    _dev(target_logits, "target_logits")
    _dev(draft_logits, "draft_logits")
    _dev(temperature, "temperature", torch.float32)
    B, K1, V = target_logits.shape
    K = K1 - 1
    if tuple(draft_logits.shape) != (B, K, V):
        raise ValueError(f"draft_logits shape {tuple(draft_logits.shape)} != {(B, K, V)}")
    dev = target_logits.device
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_accept_prob is None and want_accept_prob:
        out_accept_prob = torch.empty((B, K), dtype=torch.float32, device=dev)
    if isinstance(workspace, str):
        workspace = _auto_workspace(B, K, V, stream) if B > 0 else None
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    st = lib().spec_sample_and_verify(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft_logits),
                                      _dtype_code(draft_logits), _ptr(temperature), B, K, V, int(seed), int(offset),
                                      _ptr(out_draft_tokens), _ptr(out_tokens), _ptr(out_count),
                                      _ptr(out_accept_prob), ws_ptr, ws_bytes, _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_sample_and_verify")
    return out_draft_tokens, out_tokens, out_count, out_accept_prob


def spec_greedy_accept(target_logits, draft_tokens, *, out_tokens=None, out_count=None, stream=None):
    """Greedy acceptance for every row.  Returns (out_tokens [B][K+1], out_count [B])."""
    torch = _torch()
    _dev(target_logits, "target_logits")
    B, K1, V = target_logits.shape
    K = K1 - 1
    _dev(draft_tokens, "draft_tokens", torch.int32)
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=dev)
    st = lib().spec_greedy_accept(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), B, K, V,
                                  _ptr(out_tokens), _ptr(out_count), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_greedy_accept")
    return out_tokens, out_count


def spec_verify_tree(target_logits, draft, node_tokens, parent, temperature, max_depth: int, seed: int,
                     offset: int, *, draft_kind, out_tokens=None, out_count=None, out_path=None,
                     sibling_rule="without_replacement", stream=None):
    """Tree verify.  target_logits/draft [B][N+1][V], node_tokens/parent int32 [B][N],
    temperature fp32 [B].  sibling_rule: "without_replacement" (children drawn without
    replacement from q) or "iid" (drawn independently; a token may repeat).
    Returns (out_tokens [B][D+1], out_count [B], out_path [B][D])."""
    torch = _torch()
    _dev(target_logits, "target_logits")
    B, N1, V = target_logits.shape
    N = N1 - 1
    dk = _kind(draft_kind)
    _dev(draft, "draft")
    _dev(node_tokens, "node_tokens", torch.int32)
    _dev(parent, "parent", torch.int32)
    _dev(temperature, "temperature", torch.float32)
    if tuple(draft.shape) != (B, N + 1, V):
        raise ValueError(f"draft shape {tuple(draft.shape)} != {(B, N + 1, V)}")
    D = int(max_depth)
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_path is None:
        out_path = torch.empty((B, D), dtype=torch.int32, device=dev)
    rules = {"without_replacement": SV_SIBLINGS_WITHOUT_REPLACEMENT, "iid": SV_SIBLINGS_IID}
    if sibling_rule not in rules:
        raise ValueError("sibling_rule must be 'without_replacement' or 'iid'")
    st = lib().spec_verify_tree_rule(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft),
                                     _dtype_code(draft), dk, _ptr(node_tokens), _ptr(parent), _ptr(temperature), B,
                                     N, V, D, rules[sibling_rule], int(seed), int(offset), _ptr(out_tokens),
                                     _ptr(out_count), _ptr(out_path), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_tree")
    return out_tokens, out_count, out_path


def spec_verify_count_invalid(out_count, *, out_invalid=None, stream=None):
    """Number of invalid batch rows (out_count == 0) of a finished verify call, counted
    on the device in stream order; returns an int32 device tensor of one element."""
    torch = _torch()
    _dev(out_count, "out_count", torch.int32)
    if out_invalid is None:
        out_invalid = torch.empty((1,), dtype=torch.int32, device=out_count.device)
    st = lib().spec_verify_count_invalid(_ptr(out_count), out_count.numel(), _ptr(out_invalid), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_count_invalid")
    return out_invalid


def spec_verify_host_sizes(B: int, K: int, V: int, *, target_dtype, draft_dtype, draft_kind):
    """(offsets of target, draft, tokens, temperature in the packed input, input bytes,
    output bytes) of spec_verify_chain_host's buffers; dtypes are torch dtypes."""
    off = (ctypes.c_size_t * 4)()
    nin, nout = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib().spec_verify_host_sizes(B, K, V, _dtype_code_of(target_dtype), _dtype_code_of(draft_dtype),
                                      _kind(draft_kind), ctypes.cast(off, ctypes.c_void_p), ctypes.byref(nin),
                                      ctypes.byref(nout))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_host_sizes")
    return tuple(off), nin.value, nout.value


def spec_verify_chain_host(h_in, d_in, h_out, d_out, B: int, K: int, V: int, seed: int, offset: int, *,
                           target_dtype, draft_dtype, draft_kind, workspace=None, stream=None):
    """One round from host memory: h_in (pinned uint8, the packed inputs of
    spec_verify_host_sizes) copied into d_in (uint8 CUDA), the chain verify, and the
    tokens [B][K+1] then counts [B] (int32) copied from d_out into h_out (pinned), all
    enqueued on the stream.  h_out holds them once the stream has passed this call."""
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    st = lib().spec_verify_chain_host(h_in.data_ptr(), _ptr(d_in), h_out.data_ptr(), _ptr(d_out),
                                      _dtype_code_of(target_dtype), _dtype_code_of(draft_dtype), _kind(draft_kind),
                                      B, K, V, int(seed), int(offset), ws_ptr, ws_bytes, _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_chain_host")


def spec_verify_rows_status(out_count, *, out_status=None, stream=None):
    """Row-status summary of a finished verify call, computed on the device in stream
    order: an int32 device tensor [3] = (the call's sv_status -- SV_ERR_TIMEOUT if a row
    has count -1, else SV_ERR_BAD_INPUT if a row has count 0, else SV_OK --, the rows
    with count 0, the rows with count -1)."""
    torch = _torch()
    _dev(out_count, "out_count", torch.int32)
    if out_status is None:
        out_status = torch.empty((3,), dtype=torch.int32, device=out_count.device)
    st = lib().spec_verify_rows_status(_ptr(out_count), out_count.numel(), _ptr(out_status), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_rows_status")
    return out_status


def rows_status(out_count, *, stream=None) -> int:
    """The sv_status of a finished verify call's rows: SV_ERR_TIMEOUT if a bounded
    device-side wait gave up on some row (count -1), SV_ERR_BAD_INPUT if some row held
    invalid data (count 0), else SV_OK.  Reads three int32 back, so it waits for the
    stream."""
    s = spec_verify_rows_status(out_count, stream=stream)
    (_torch().cuda.current_stream() if stream is None else stream).synchronize()
    return int(s[0].cpu().item())


def spec_tree_mask(parent, *, out_mask=None, out_depth=None, out_valid=None, stream=None):
    """Ancestor-or-self attention mask of each draft tree.  parent int32 [B][N].
    Returns (out_mask int32 [B][N][ceil(N/32)] holding the uint32 bit words, out_depth
    int32 [B][N], out_valid int32 [B])."""
    torch = _torch()
    _dev(parent, "parent", torch.int32)
    B, N = parent.shape
    W = (N + 31) // 32
    dev = parent.device
    if out_mask is None:
        out_mask = torch.empty((B, N, W), dtype=torch.int32, device=dev)
    if out_depth is None:
        out_depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_valid is None:
        out_valid = torch.empty((B,), dtype=torch.int32, device=dev)
    st = lib().spec_tree_mask(_ptr(parent), B, N, _ptr(out_mask), _ptr(out_depth), _ptr(out_valid),
                              _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_tree_mask")
    return out_mask, out_depth, out_valid


def spec_kv_compact(kv_buffers, path, count, base=None, *, stream=None):
    """Move each batch row's accepted tree nodes' cache rows to the front, in place.
    kv_buffers: CUDA tensors of one dtype and identical shape [B][planes][rows][width]
    and strides (any strided view whose last dimension is contiguous, e.g. a
    [B][rows][heads][dim] cache permuted to [B][heads][rows][dim]).  path int32
    [B][D] and count int32 [B] as spec_verify_tree returns them; base int32 [B] (the
    cache row of tree node 0) or None for 0."""
    torch = _torch()
    bufs = list(kv_buffers)
    if not bufs:
        raise ValueError("kv_buffers is empty")
    t0 = bufs[0]
    for t in bufs:
        if not t.is_cuda or t.dim() != 4 or t.shape != t0.shape or t.stride() != t0.stride() or t.dtype != t0.dtype:
            raise ValueError("kv_buffers must be CUDA tensors [B][planes][rows][width] of one shape, stride and dtype")
        if t.stride(3) != 1:
            raise ValueError("the last dimension of every kv buffer must be contiguous")
    _dev(path, "path", torch.int32)
    _dev(count, "count", torch.int32)
    _dev(base, "base", torch.int32)
    B, H, R, Wd = t0.shape
    es = t0.element_size()
    arr = (ctypes.c_void_p * len(bufs))(*[t.data_ptr() for t in bufs])
    st = lib().spec_kv_compact(arr, len(bufs), t0.stride(0) * es, t0.stride(1) * es, H, t0.stride(2) * es,
                               Wd * es, R, _ptr(path), _ptr(count), _ptr(base), B, path.shape[1],
                               _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_kv_compact")
