"""Shared helpers for the GPU parity tests: move synthetic workloads to the device,
run the library and the oracle on the same inputs, compare element by element.

Parity rule: tokens and counts are bit-exact, except on rows where the oracle saw a
decision within MARGIN of its boundary (|r - p/q| for an acceptance, the distance
from u*Z to the nearest CDF boundary, in probability mass, for a draw): fp32 on the
device may legitimately decide those differently from fp64.  Such rows are
counted.  Acceptance probabilities agree within AP_TOL absolute.
"""
import numpy as np

import oracle

MARGIN = 1e-5
AP_TOL = 1e-5


def to_dev(a):
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def kind_name(dk):
    return "probs" if dk == oracle.DRAFT_PROBS else "logits"


def gpu_chain(w, seed=None, offset=None):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    seed = w["seed"] if seed is None else seed
    offset = w["offset"] if offset is None else offset
    t, d = to_dev(w["target"]), to_dev(w["draft"])
    toks, temps = to_dev(w["tokens"].astype(np.int32)), to_dev(w["temperature"].astype(np.float32))
    ot, oc, ap = sv.spec_verify_chain(t, d, toks, temps, seed, offset, draft_kind=kind_name(w["draft_kind"]),
                                      want_accept_prob=True)
    torch.cuda.synchronize()
    return dict(tokens=ot.cpu().numpy(), count=oc.cpu().numpy(), accept_prob=ap.cpu().numpy())


def oracle_chain(w, seed=None, offset=None, rows=None):
    seed = w["seed"] if seed is None else seed
    offset = w["offset"] if offset is None else offset
    if rows is None:
        return oracle.verify_chain(w["target"], w["draft"], w["tokens"], w["temperature"], seed, offset,
                                   draft_kind=w["draft_kind"])
    rows = np.asarray(rows)
    return oracle.verify_chain(w["target"][rows], None if w["draft"] is None else w["draft"][rows],
                               w["tokens"][rows], w["temperature"][rows], seed, offset,
                               draft_kind=w["draft_kind"], row_id=rows.astype(np.int32))


RULE_NAMES = {oracle.SIBLINGS_WOR: "without_replacement", oracle.SIBLINGS_IID: "iid"}


def gpu_tree(w, seed=None, offset=None, sibling_rule=oracle.SIBLINGS_WOR):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    seed = w["seed"] if seed is None else seed
    offset = w["offset"] if offset is None else offset
    ot, oc, op = sv.spec_verify_tree(to_dev(w["target"]), to_dev(w["draft"]),
                                     to_dev(w["node_tokens"].astype(np.int32)), to_dev(w["parent"].astype(np.int32)),
                                     to_dev(w["temperature"].astype(np.float32)), w["max_depth"], seed, offset,
                                     draft_kind=kind_name(w["draft_kind"]), sibling_rule=RULE_NAMES[sibling_rule])
    torch.cuda.synchronize()
    return dict(tokens=ot.cpu().numpy(), count=oc.cpu().numpy(), path=op.cpu().numpy())


def oracle_tree(w, seed=None, offset=None, rows=None, sibling_rule=oracle.SIBLINGS_WOR):
    seed = w["seed"] if seed is None else seed
    offset = w["offset"] if offset is None else offset
    sel = slice(None) if rows is None else np.asarray(rows)
    rid = None if rows is None else np.asarray(rows, np.int32)
    return oracle.verify_tree(w["target"][sel], w["draft"][sel], w["node_tokens"][sel], w["parent"][sel],
                              w["temperature"][sel], w["max_depth"], seed, offset, draft_kind=w["draft_kind"],
                              row_id=rid, sibling_rule=sibling_rule)


def compare(gpu, ora, rows=None, keys=("tokens", "count")):
    """Assert the parity rule; returns the number of excused (near-margin) rows."""
    sel = slice(None) if rows is None else np.asarray(rows)
    g = {k: v[sel] for k, v in gpu.items()}
    same = np.ones(len(ora["count"]), bool)
    for k in keys:
        a, b = g[k], ora[k]
        same &= (a.reshape(len(a), -1) == b.reshape(len(b), -1)).all(1)
    bad = np.nonzero(~same)[0]
    unexcused = [int(i) for i in bad if not ora["margin"][i] < MARGIN]
    assert not unexcused, (f"{len(unexcused)} rows differ with margin >= {MARGIN}: rows {unexcused[:8]}; "
                           f"gpu {[(g['tokens'][i].tolist(), int(g['count'][i])) for i in unexcused[:3]]} "
                           f"oracle {[(ora['tokens'][i].tolist(), int(ora['count'][i])) for i in unexcused[:3]]}")
    if "accept_prob" in g and "accept_prob" in ora:
        ga, oa = g["accept_prob"][same], ora["accept_prob"][same]
        evaluated = oa >= 0
        assert np.array_equal(ga >= 0, evaluated), "accept_prob: evaluated positions differ"
        if evaluated.any():
            err = np.abs(ga[evaluated].astype(np.float64) - oa[evaluated])
            assert err.max() <= AP_TOL, f"accept_prob error {err.max():.3g} > {AP_TOL}"
    return len(bad)
