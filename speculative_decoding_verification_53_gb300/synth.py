"""Seeded synthetic inputs for the verify/accept step.

This module produces INPUTS only: target logits, the draft distribution, the
drafted tokens (or draft trees), temperatures.  It serves the CUDA path, the
CPU oracle, the tests and the benchmark alike, and holds none of the verify
rule's arithmetic (no acceptance test, no residual, no draw over the target).
The draft model is out of scope, so a stand-in drafter lives here: it turns
noisy copies of the target logits into a draft distribution (a softmax, for
workloads that hand the verifier probabilities), samples the drafted tokens
from it and grows best-first draft trees from it.

Workloads (sizes and value distributions from the five verify workloads):
  tiny_chain        B=1, K=4, V=1024 (or V=8), fp32; target ~ N(0, 2^2),
                    draft logits = target + N(0, 0.5^2), T = 1.
  single_stream     B=1, K=5, V=128256, T=0.8; bf16 target ~ N(0, 3^2) plus a
                    Zipf(1.1) log-prior over token ids; draft probabilities
                    fp32 = softmax(target + N(0, 1^2)) (no temperature).
  mixed_batch       B=64, K=5, V=32000, bf16 target ~ N(0, 2^2), bf16 draft
                    logits = target + N(0, sigma_b^2), sigma_b in {0.25, 1, 4}
                    by b mod 3; T_b = 0 (greedy) for even b, 1.0 for odd b.
  tree              B=16, V=128256, N=60 nodes, depth <= 6, top-3 branching by
                    draft probability, best-first by cumulative draft
                    probability, nodes renumbered breadth-first with siblings
                    sorted by draft probability; bf16 logits as single_stream,
                    draft logits = target + N(0, 1^2).
  large_batch       B=256, K=8, V=152064, bf16 target as single_stream, bf16
                    draft logits = target + N(0, sigma^2); T in {0, 0.7, 1.5}.

Every batch row b draws from its own generator ``default_rng([seed, b])``, so
any subset of rows can be regenerated alone.  Greedy rows (T <= 0) draft by
argmax of the draft logits; sampling rows draw x_k from the draft
distribution by inverse CDF in float64.
"""
from __future__ import annotations

import heapq

import numpy as np

DRAFT_PROBS, DRAFT_LOGITS = 0, 1


# ----------------------------------------------------------------- encoding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even) and return the bit patterns
    as uint16.  NaN stays NaN; infinities stay infinite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    rounded = ((bits.astype(np.uint64) + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded[nan] = 0x7FC0
    return rounded


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_f32(logits: np.ndarray) -> np.ndarray:
    """Logits as float32 values, whatever their storage (float32 or bf16 bits)."""
    return bf16_bits_to_f32(logits) if logits.dtype == np.uint16 else np.asarray(logits, np.float32)


# ---------------------------------------------------------- drafter stand-in

def _draft_probs64(row_logits: np.ndarray, temperature: float) -> np.ndarray:
    z = np.asarray(row_logits, np.float64) / temperature
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def draft_tokens_from_logits(rng, draft_logits_f32: np.ndarray, temperature: float) -> np.ndarray:
    """Drafted tokens for one batch row: [K][V] draft logits -> [K] tokens.
    Greedy drafting (argmax) for temperature <= 0, else inverse-CDF sampling from
    softmax(logits / T)."""
    K = draft_logits_f32.shape[0]
    out = np.empty(K, np.int32)
    for k in range(K):
        if not temperature > 0:
            out[k] = int(np.argmax(draft_logits_f32[k]))
        else:
            c = np.cumsum(_draft_probs64(draft_logits_f32[k], temperature))
            out[k] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), c.size - 1)
    return out


def draft_tokens_from_probs(rng, probs: np.ndarray) -> np.ndarray:
    K = probs.shape[0]
    out = np.empty(K, np.int32)
    for k in range(K):
        c = np.cumsum(probs[k].astype(np.float64))
        out[k] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), c.size - 1)
    return out


def zipf_log_prior(V: int, s: float = 1.1) -> np.ndarray:
    """log of an unnormalised Zipf(s) law over token ids: -s * ln(i + 1)."""
    return (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)


# --------------------------------------------------------------- workloads

def tiny_chain(seed: int, V: int = 1024, K: int = 4, B: int = 1, temperature: float = 1.0,
               sigma: float = 0.5, scale: float = 2.0):
    """fp32 chain workload: target ~ N(0, scale^2), draft logits = target + N(0, sigma^2)."""
    target = np.empty((B, K + 1, V), np.float32)
    draft = np.empty((B, K, V), np.float32)
    tokens = np.empty((B, K), np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b])
        target[b] = rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(scale)
        draft[b] = target[b, :K] + rng.standard_normal((K, V), dtype=np.float32) * np.float32(sigma)
        tokens[b] = draft_tokens_from_logits(rng, draft[b], temperature)
    return dict(kind="chain", target=target, draft=draft, draft_kind=DRAFT_LOGITS, tokens=tokens,
                temperature=np.full(B, temperature, np.float32), seed=seed, offset=0)


def single_stream(seed: int, V: int = 128256, K: int = 5, B: int = 1, temperature: float = 0.8):
    """bf16 target with a Zipf(1.1) prior; fp32 draft probabilities softmax(target + N(0,1))."""
    prior = zipf_log_prior(V)
    target = np.empty((B, K + 1, V), np.uint16)
    draft = np.empty((B, K, V), np.float32)
    tokens = np.empty((B, K), np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b])
        t = f32_to_bf16_bits(rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(3.0) + prior)
        target[b] = t
        noisy = bf16_bits_to_f32(t[:K]) + rng.standard_normal((K, V), dtype=np.float32)
        for k in range(K):
            draft[b, k] = _draft_probs64(noisy[k], 1.0).astype(np.float32)
        tokens[b] = draft_tokens_from_probs(rng, draft[b])
    return dict(kind="chain", target=target, draft=draft, draft_kind=DRAFT_PROBS, tokens=tokens,
                temperature=np.full(B, temperature, np.float32), seed=seed, offset=0)


def mixed_batch(seed: int, B: int = 64, K: int = 5, V: int = 32000):
    """bf16 target ~ N(0, 2^2) and bf16 draft logits; even rows greedy, odd rows T=1;
    draft noise sigma_b = (0.25, 1, 4)[b mod 3]."""
    target = np.empty((B, K + 1, V), np.uint16)
    draft = np.empty((B, K, V), np.uint16)
    tokens = np.empty((B, K), np.int32)
    temps = np.empty(B, np.float32)
    for b in range(B):
        rng = np.random.default_rng([seed, b])
        sigma = (0.25, 1.0, 4.0)[b % 3]
        temps[b] = 0.0 if b % 2 == 0 else 1.0
        t = f32_to_bf16_bits(rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(2.0))
        target[b] = t
        d = f32_to_bf16_bits(bf16_bits_to_f32(t[:K]) +
                             rng.standard_normal((K, V), dtype=np.float32) * np.float32(sigma))
        draft[b] = d
        tokens[b] = draft_tokens_from_logits(rng, bf16_bits_to_f32(d), float(temps[b]))
    return dict(kind="chain", target=target, draft=draft, draft_kind=DRAFT_LOGITS, tokens=tokens,
                temperature=temps, seed=seed, offset=0)


def large_batch(seed: int, temperature: float, sigma: float = 1.0, B: int = 256, K: int = 8,
                V: int = 152064):
    """bf16 target (N(0, 3^2) + Zipf prior) and bf16 draft logits = target + N(0, sigma^2)."""
    prior = zipf_log_prior(V)
    target = np.empty((B, K + 1, V), np.uint16)
    draft = np.empty((B, K, V), np.uint16)
    tokens = np.empty((B, K), np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b])
        t = f32_to_bf16_bits(rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(3.0) + prior)
        target[b] = t
        d = f32_to_bf16_bits(bf16_bits_to_f32(t[:K]) +
                             rng.standard_normal((K, V), dtype=np.float32) * np.float32(sigma))
        draft[b] = d
        tokens[b] = draft_tokens_from_logits(rng, bf16_bits_to_f32(d), temperature)
    return dict(kind="chain", target=target, draft=draft, draft_kind=DRAFT_LOGITS, tokens=tokens,
                temperature=np.full(B, temperature, np.float32), seed=seed, offset=0)


def best_first_tree(draft_rows_f32: np.ndarray, n_nodes: int, max_depth: int, branch: int,
                    temperature: float = 1.0):
    """Grow a draft tree best-first by cumulative draft log-probability.

    ``draft_rows_f32[j]`` is the draft logit row of the j-th created node (row 0 is
    the root).  Each node offers its top-``branch`` tokens as children.  Returns
    (tokens, parent, row_of_node) in breadth-first order with siblings sorted by
    draft probability (descending), so parent[i] < i; ``row_of_node[i]`` is the
    creation row of node i (its own next-token row)."""
    def top_children(row_idx, base_score):
        lp = np.log(_draft_probs64(draft_rows_f32[row_idx], temperature))
        top = np.argsort(-lp, kind="stable")[:branch]
        return [(base_score + lp[t], int(t), float(lp[t])) for t in top]

    heap, counter = [], 0
    created = []  # (creation parent id or -1, token, depth, logq)
    for score, tok, lq in top_children(0, 0.0):
        heapq.heappush(heap, (-score, counter, -1, tok, 1, lq))
        counter += 1
    while heap and len(created) < n_nodes:
        negs, _, par, tok, depth, lq = heapq.heappop(heap)
        created.append((par, tok, depth, lq))
        cid = len(created) - 1
        if depth < max_depth and cid + 1 < draft_rows_f32.shape[0]:
            for score, ctok, clq in top_children(cid + 1, -negs):
                heapq.heappush(heap, (-score, counter, cid, ctok, depth + 1, clq))
                counter += 1
    kids = {}
    for cid, (par, tok, depth, lq) in enumerate(created):
        kids.setdefault(par, []).append(cid)
    order, queue = [], [-1]
    while queue:
        nxt = []
        for node in queue:
            ch = sorted(kids.get(node, []), key=lambda c: (-created[c][3], c))
            order.extend(ch)
            nxt.extend(ch)
        queue = nxt
    new_id = {cid: i for i, cid in enumerate(order)}
    tokens = np.array([created[c][1] for c in order], np.int32)
    parent = np.array([new_id[created[c][0]] if created[c][0] >= 0 else -1 for c in order], np.int32)
    row_of_node = np.array([c + 1 for c in order], np.int64)
    return tokens, parent, row_of_node


def tree(seed: int, temperature: float = 1.0, B: int = 16, N: int = 60, V: int = 128256,
         max_depth: int = 6, branch: int = 3, sigma: float = 1.0):
    """Tree workload: per batch row a best-first draft tree of N nodes; target/draft
    rows laid out [B][N+1][V] with row 0 the root and row i+1 the row after node i."""
    prior = zipf_log_prior(V)
    target = np.empty((B, N + 1, V), np.uint16)
    draft = np.empty((B, N + 1, V), np.uint16)
    tokens = np.empty((B, N), np.int32)
    parent = np.empty((B, N), np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b])
        t = f32_to_bf16_bits(rng.standard_normal((N + 1, V), dtype=np.float32) * np.float32(3.0) + prior)
        d = f32_to_bf16_bits(bf16_bits_to_f32(t) +
                             rng.standard_normal((N + 1, V), dtype=np.float32) * np.float32(sigma))
        tk, par, rows = best_first_tree(bf16_bits_to_f32(d), N, max_depth, branch)
        perm = np.concatenate([[0], rows])
        target[b] = t[perm]
        draft[b] = d[perm]
        tokens[b] = tk
        parent[b] = par
    return dict(kind="tree", target=target, draft=draft, draft_kind=DRAFT_LOGITS, node_tokens=tokens,
                parent=parent, temperature=np.full(B, temperature, np.float32), max_depth=max_depth,
                seed=seed, offset=0)


def chain_as_tree(w: dict) -> dict:
    """Re-express a chain workload as a tree whose parent array is the chain
    (parent[i] = i - 1).  The draft gains an unused last row."""
    target, draft = w["target"], w["draft"]
    B, K1, V = target.shape
    K = K1 - 1
    pad = np.zeros((B, 1, V), draft.dtype)
    parent = np.tile(np.arange(-1, K - 1, dtype=np.int32), (B, 1))
    return dict(kind="tree", target=target, draft=np.concatenate([draft, pad], axis=1),
                draft_kind=w["draft_kind"], node_tokens=w["tokens"].copy(), parent=parent,
                temperature=w["temperature"].copy(), max_depth=K, seed=w["seed"], offset=w["offset"])


def redraw_tokens(w: dict, temperature: float, seed: int) -> dict:
    """The same chain logits with drafted tokens (and temperatures) redrawn for another
    temperature; row b draws from ``default_rng([seed, b, 1])``."""
    B, K = w["tokens"].shape
    tokens = np.empty_like(w["tokens"])
    for b in range(B):
        rng = np.random.default_rng([seed, b, 1])
        if w["draft_kind"] == DRAFT_PROBS:
            tokens[b] = draft_tokens_from_probs(rng, w["draft"][b])
        else:
            tokens[b] = draft_tokens_from_logits(rng, as_f32(w["draft"][b]), temperature)
    out = dict(w)
    out["tokens"] = tokens
    out["temperature"] = np.full(B, temperature, np.float32)
    return out


# ------------------------------------------------------------ tree shapes and KV caches

def random_parents(seed: int, B: int, N: int, shape: str = "bfs", branch: int = 3,
                   max_depth: int = 6) -> np.ndarray:
    """Parent arrays [B][N] with parent[i] in {-1} u [0, i).

    shape: "bfs"    breadth-first tree, up to ``branch`` children a node and depth
                    <= ``max_depth`` (the draft-tree shape), a random fan-out per node;
           "random" parent[i] uniform over {-1, 0, .., i-1} (deep, irregular);
           "chain"  parent[i] = i - 1;  "star"  every node a child of the root."""
    out = np.empty((B, N), np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b, 7])
        if shape == "chain":
            out[b] = np.arange(-1, N - 1)
        elif shape == "star":
            out[b] = -1
        elif shape == "random":
            out[b] = [int(rng.integers(-1, i)) if i > 0 else -1 for i in range(N)]
        else:
            par, depth = [], []
            frontier = [(-1, 0)]          # (node, depth); -1 is the root
            head = 0
            while len(par) < N:
                if head >= len(frontier):  # every node at max depth: restart at the root
                    frontier.append((-1, 0))
                node, d = frontier[head]
                head += 1
                if d >= max_depth:
                    continue
                for _ in range(int(rng.integers(1, branch + 1))):
                    if len(par) == N:
                        break
                    par.append(node)
                    depth.append(d + 1)
                    frontier.append((len(par) - 1, d + 1))
            out[b] = par
    return out


def accepted_paths(seed: int, parent: np.ndarray, max_depth: int):
    """A tree-verify-shaped result for each batch row: a random node's root-to-node
    path (node indices, -1 padded to ``max_depth``) and count = path length + 1.
    Rows whose chosen node is deeper than ``max_depth`` take its ancestor at that depth."""
    B, N = parent.shape
    path = np.full((B, max_depth), -1, np.int32)
    count = np.empty(B, np.int32)
    for b in range(B):
        rng = np.random.default_rng([seed, b, 11])
        chain = []
        j = int(rng.integers(-1, N))     # -1: nothing accepted
        while j >= 0:
            chain.append(j)
            j = int(parent[b, j])
        chain = chain[::-1][:max_depth]
        path[b, :len(chain)] = chain
        count[b] = len(chain) + 1
    return path, count


def kv_cache(seed: int, n_buffers: int, B: int, planes: int, rows: int, row_bytes: int) -> np.ndarray:
    """Random bytes shaped [n_buffers][B][planes][rows][row_bytes] (one buffer per
    layer and K/V; a plane is a KV head; a row is one token's head vector)."""
    rng = np.random.default_rng([seed, 13])
    return rng.integers(0, 256, (n_buffers, B, planes, rows, row_bytes), dtype=np.uint8)


def redraw_children_iid(w: dict, seed: int) -> dict:
    """The tree of ``w`` with every node's token redrawn independently from its parent's
    draft distribution (the row the node was proposed from), so siblings may repeat:
    the drafts of a multi-draft verifier that samples each child i.i.d. from q.
    Draft logits are turned into q with the row's temperature (1 for greedy rows)."""
    out = dict(w)
    toks = w["node_tokens"].copy()
    B, N = toks.shape
    for b in range(B):
        rng = np.random.default_rng([seed, b, 17])
        T = float(w["temperature"][b]) if w["temperature"][b] > 0 else 1.0
        cache = {}
        for i in range(N):
            row = int(w["parent"][b, i]) + 1
            if row not in cache:
                d = w["draft"][b, row]
                d = bf16_bits_to_f32(d) if d.dtype == np.uint16 else d.astype(np.float32)
                if w["draft_kind"] == 0:
                    q = d.astype(np.float64)
                else:
                    z = d.astype(np.float64) / T
                    q = np.exp(z - z.max())
                q = q / q.sum()
                cache[row] = np.cumsum(q)
            cdf = cache[row]
            toks[b, i] = min(int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right")), cdf.size - 1)
    out["node_tokens"] = toks
    return out
