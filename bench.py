#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verify step on GB300.

Default workload (the headline metric): single-stream chain verify, B=1, K=5,
V=128256, T=0.8, bf16 target logits, fp32 draft probabilities.  One step is one
verify round (the whole path: softmax statistics, acceptance, first rejection,
replacement or bonus draw) of one batch.  ROUNDS distinct rounds (default 64,
about 262 MB, more than the 129 MB L2) stay resident in HBM and the steps cycle
through them; steps are replayed from CUDA graphs so that host launch gaps do
not enter the device timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload single_stream|large_batch|mixed_batch|sample_verify|tree|tree_iid|tree_mask|kv_compact]

tree_mask and kv_compact time the steps on either side of a tree verify (the
ancestor attention mask of each draft tree; moving the accepted branch's KV-cache
rows to the front) with their own metric and unit.

Prints one JSON line (rank 0).  `value` is verify rows/s over all ranks (under
torchrun every rank is an independent replica on its own rows; the time is the
slowest rank's); `roofline` relates the kernel's algorithmic bytes per launch
(the rows the rule needs: target rows up to the first rejection, gathered draft
entries, the draft row of the rejected position) to its event-timed duration,
and `roofline.traffic` is the DRAM bytes per launch from the committed ncu
summary of that kernel (null once the kernel's sources have changed); `e2e` is
the same metric through the public API with host buffers (copies inside the
timed region); `cpu_baseline` is the fp64 oracle on a bounded sample, single
thread; `acceptance` (chain workloads with sampling rows) is the mean of the
library's min(1, p/q) per drafted position, from untimed calls after the timed
region.  With the default single-stream workload the line also carries
`workloads`: the large batch at T = 0, 0.7 and 1.5, the mixed batch and the tree,
each timed the same way.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rows/s and achieved HBM GB/s vs GB300 peak at V=128256, K=5"
UNIT = "verify rows/s"
# streams that take the end-to-end chain steps in turn (a copy's fixed start-up latency overlaps
# the steps before it; past four the host-to-device link is the bound)
E2E_STREAMS = 4
FALLBACK_HBM_GBS = 6800.0
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ------------------------------------------------------------------ inputs

def large_batch_at(w, T):
    """The large batch at temperature T: the T = 0.7 workload's logits, with the drafted
    tokens redrawn at T (the same inputs whether T is the run's workload or a side line)."""
    from speculative_decoding_verification_53_gb300 import synth
    return w if T == 0.7 else synth.redraw_tokens(w, T, seed=100 + int(T * 10))


def make_workload(name: str, rank: int, rounds: int, batch: int = 0, temperature=None):
    from speculative_decoding_verification_53_gb300 import synth
    seed = 1000 + rank
    if name == "single_stream":
        w = synth.single_stream(seed=seed, B=rounds)  # row r = round r (B=1 per step)
        return dict(w, per_step_rows=1, desc="single-stream chain verify B=1 K=5 V=128256 T=0.8, "
                                             "bf16 target logits, fp32 draft probabilities")
    if name == "large_batch":
        B = batch or 256
        T = 0.7 if temperature is None else temperature
        w = large_batch_at(synth.large_batch(seed=seed, temperature=0.7, sigma=1.0, B=B), T)
        return dict(w, per_step_rows=B, desc=f"large-batch chain verify B={B} K=8 V=152064 T={T:g}, "
                                             "bf16 target and draft logits, draft noise sigma=1")
    if name == "mixed_batch":
        w = synth.mixed_batch(seed=seed)
        return dict(w, per_step_rows=64, desc="mixed greedy/sampling chain verify B=64 K=5 V=32000, bf16 logits")
    if name == "sample_verify":
        w = synth.mixed_batch(seed=seed)
        return dict(w, per_step_rows=64, sample=True,
                    desc="draft sampling + chain verify in one call, B=64 K=5 V=32000, bf16 logits, "
                         "greedy/sampling rows mixed")
    if name == "tree":
        w = synth.tree(seed=seed, temperature=1.0)
        return dict(w, per_step_rows=16, desc="tree verify B=16 N=60 depth<=6 V=128256 T=1, bf16 logits")
    if name == "tree_iid":
        w = synth.redraw_children_iid(synth.tree(seed=seed, temperature=1.0), seed=seed)
        return dict(w, per_step_rows=16, sibling_rule="iid",
                    desc="multi-draft tree verify B=16 N=60 depth<=6 V=128256 T=1, children drawn i.i.d. from q "
                         "(i.i.d. sibling rule), bf16 logits")
    raise ValueError(name)


def to_dev(a, device):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def pinned(a):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


# ----------------------------------------------------------------- helpers

# translation unit each profiled kernel is compiled from
KERNEL_SOURCES = {"chain_spec_kernel": "sv_chain_spec.cu", "chain_staged_kernel": "sv_chain_staged.cu",
                  "tree_staged_kernel": "sv_tree_staged.cu", "draft_sample_staged_kernel": "sv_sample.cu",
                  "tree_mask_kernel": "sv_tree_kv.cu", "kv_compact_kernel": "sv_tree_kv.cu"}


def kernel_source_hash(kernel: str = None) -> str:
    """sha256 prefix of the device sources a kernel is compiled from: its translation
    unit and the package's internal headers (.cuh, .h).  With no kernel (or one not
    listed), every source file of the package and of include/."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "speculative_decoding_verification_53_gb300", "csrc")
    if kernel in KERNEL_SOURCES:
        files = [os.path.join(pkg, f) for f in sorted(os.listdir(pkg)) if f.endswith((".cuh", ".h"))]
        files.append(os.path.join(pkg, KERNEL_SOURCES[kernel]))
    else:
        files = [os.path.join(d, f) for d in (pkg, os.path.join(ROOT, "include")) for f in sorted(os.listdir(d))]
    for path in files:
        with open(path, "rb") as fh:
            h.update(os.path.basename(path).encode() + fh.read())
    return h.hexdigest()[:16]


def slowest_rank_ms(elapsed_ms: float, world: int, device) -> float:
    """Length of the timed region on the slowest rank: the max over ranks (every rank
    gets it).  `device` is where the collective's tensor lives (CUDA under NCCL, CPU
    under gloo)."""
    import torch
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Units all ranks processed (each its own, the same count per step) per second of
    the slowest rank's timed region."""
    return units_per_step * steps * world / (max_ms / 1e3)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if j.get("hbm_gbs"):
            return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(workload: str, default_size: bool = True):
    """DRAM bytes per launch of the timed kernel from the committed ncu summary for this
    workload (profiles/<kernel>_<workload>.md), if that kernel's sources still hash to the
    value recorded there and the run uses the workload's default size and temperature
    (the summaries describe that configuration); else None.  Returns (bytes, summary
    path, kernel name)."""
    import glob
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_{workload}.md"))):
        text = open(path).read()
        m = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        hm = re.search(r"^kernel_source_sha:\s*([0-9a-f]+)", text, re.M)
        km = re.search(r"^kernel:\s*(\S+)", text, re.M)
        kernel = km.group(1) if km else None
        if not m or not hm or hm.group(1) != kernel_source_hash(kernel) or not default_size:
            return None, os.path.relpath(path, ROOT), kernel
        return float(m.group(1)), os.path.relpath(path, ROOT), kernel
    return None, None, None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes_chain(w, rows, counts):
    """Bytes the rule needs for the given rounds: target rows 0..j, the gathered draft
    entries (probabilities) or draft rows 0..min(j, K-1) (logits), the draft row of a
    rejected position, tokens, temperature and the outputs.  j = count - 1."""
    target, draft = w["target"], w["draft"]
    _, K1, V = target.shape
    K = K1 - 1
    tb = V * target.dtype.itemsize
    db = V * draft.dtype.itemsize
    total = 0
    for b, cnt in zip(rows, counts):
        j = int(cnt) - 1
        greedy = not (w["temperature"][b] > 0)
        total += (j + 1) * tb + K * 4 + 4 + (K + 1) * 4 + 4
        if greedy:
            continue
        evaluated = min(j, K - 1) + 1 if K > 0 else 0
        if w["draft_kind"] == 0:  # probabilities: gathered entries, plus the rejected row
            total += evaluated * 4 + (db if j < K else 0)
        else:  # logits: every evaluated draft row is streamed for its statistics
            total += evaluated * db
    return total


def algorithmic_bytes_tree(w, counts, paths):
    target = w["target"]
    B, N1, V = target.shape
    tb = V * target.dtype.itemsize
    db = V * w["draft"].dtype.itemsize
    total = 0
    for b in range(B):
        visited = int(counts[b])  # root plus accepted nodes: one row each
        total += visited * tb + N1 * 8 + 4 + 4
        if w["temperature"][b] > 0:
            par = w["parent"][b]
            nodes = [-1] + [int(x) for x in paths[b][: visited - 1]]
            total += sum(db for n in nodes if (par == n).any())
    return total


# ---------------------------------------------------------------- our arm

L2_FLUSH_BYTES = 512 << 20  # read right before every timed region (the L2 holds 129 MB)


def dense_bytes_chain(w, rows):
    """Bytes of every row the verify could read, whatever the decisions: all K+1 target
    rows, plus the K draft rows of sampling rows (logits), or the K gathered draft
    probabilities and one draft row (probabilities)."""
    target, draft = w["target"], w["draft"]
    _, K1, V = target.shape
    K = K1 - 1
    tb, db = V * target.dtype.itemsize, V * draft.dtype.itemsize
    total = 0
    for b in rows:
        total += K1 * tb
        if w["temperature"][b] > 0 and K > 0:
            total += K * db if w["draft_kind"] == 1 else K * 4 + db
    return total


def dense_bytes_tree(w):
    """Every target row of every tree (the rows a level-by-level evaluation would read)."""
    t = w["target"]
    return t.shape[0] * t.shape[1] * t.shape[2] * t.dtype.itemsize


class Timed:
    """One workload resident on the device, its steps captured in CUDA graphs."""

    def __init__(self, w, device, stream, steps, warmup, seed=17, dev_inputs=None):
        import torch
        import speculative_decoding_verification_53_gb300 as sv
        self.w, self.device, self.stream, self.steps = w, device, stream, steps
        self.tree = w["kind"] == "tree"
        self.sample = bool(w.get("sample"))
        rule = w.get("sibling_rule", "without_replacement")
        rows = w["per_step_rows"]
        if dev_inputs is None:
            dev_inputs = {k: to_dev(w[k], device) for k in ("target", "draft")}
        dt, dd = dev_inputs["target"], dev_inputs["draft"]
        if self.tree:
            dtok, dpar = to_dev(w["node_tokens"], device), to_dev(w["parent"], device)
        else:
            dtok = to_dev(w["tokens"], device)
        dtemp = to_dev(w["temperature"], device)
        kind = "probs" if w["draft_kind"] == 0 else "logits"
        self.n_inputs = dt.shape[0] // rows
        self.resident_bytes = int(dt.numel() * dt.element_size() + dd.numel() * dd.element_size())
        chunk = min(steps, 1000)
        self.chunk = chunk
        if self.tree:
            D = w["max_depth"]
            out_t = torch.empty((chunk, rows, D + 1), dtype=torch.int32, device=device)
            self.out_c = torch.empty((chunk, rows), dtype=torch.int32, device=device)
            self.out_p = torch.empty((chunk, rows, D), dtype=torch.int32, device=device)
        else:
            K_ = w["tokens"].shape[1]
            out_t = torch.empty((chunk, rows, K_ + 1), dtype=torch.int32, device=device)
            self.out_c = torch.empty((chunk, rows), dtype=torch.int32, device=device)
            out_x = torch.empty((chunk, rows, K_), dtype=torch.int32, device=device)
            ws_bytes = sv.spec_verify_workspace_size(rows, K_, w["target"].shape[2])
            ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=device)
        n_inputs = self.n_inputs
        self._chain_inputs = None if (self.tree or self.sample) else (dt, dd, dtok, dtemp, kind, seed)
        # every tensor the captured graphs read or write stays referenced by this object:
        # a graph holds raw device pointers only, so a tensor that went out of scope here
        # would be freed and its memory reused while the graphs still run on it
        self._graph_tensors = [dt, dd, dtok, dtemp, out_t] + ([dpar, self.out_p] if self.tree else [out_x, ws])

        def step(i, slot):
            r = (i % n_inputs) * rows
            sl = slice(r, r + rows)
            if self.tree:
                sv.spec_verify_tree(dt[sl], dd[sl], dtok[sl], dpar[sl], dtemp[sl], D, seed, i, draft_kind=kind,
                                    out_tokens=out_t[slot], out_count=self.out_c[slot], out_path=self.out_p[slot],
                                    sibling_rule=rule)
            elif self.sample:
                sv.spec_sample_and_verify(dt[sl], dd[sl], dtemp[sl], seed, i, out_draft_tokens=out_x[slot],
                                          out_tokens=out_t[slot], out_count=self.out_c[slot], workspace=ws)
            else:
                sv.spec_verify_chain(dt[sl], dd[sl], dtok[sl], dtemp[sl], seed, i, draft_kind=kind,
                                     out_tokens=out_t[slot], out_count=self.out_c[slot], workspace=ws)

        with torch.cuda.stream(stream):
            for i in range(max(warmup, 3)):
                step(i, i % chunk)
        torch.cuda.synchronize(device)

        def capture(nsteps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(nsteps):
                    step(i, i)
            return g

        self.reps, self.rem = divmod(steps, chunk)
        self.g_main = capture(chunk) if self.reps else None
        self.g_rem = capture(self.rem) if self.rem else None
        for g in (self.g_main, self.g_rem):  # untimed: every captured step runs once
            if g is not None:
                g.replay()
        torch.cuda.synchronize(device)
        # L2 flush by a read of a 512 MB buffer (a reduction): it evicts the inputs without
        # leaving dirty lines whose write-back would compete with the timed kernels
        self.flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def run(self, world, clocks_gpu):
        """Times `steps` steps: barrier, synchronize, an L2 flush (a 512 MB read), then
        the graph replays between two CUDA events on the launching stream."""
        import torch
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(clocks_gpu) as clocks:
            t_wall = time.time()
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize(self.device)
            with torch.cuda.stream(self.stream):
                self.flush_sum = self.flush.sum()
            start.record(self.stream)
            for _ in range(self.reps):
                self.g_main.replay()
            if self.g_rem is not None:
                self.g_rem.replay()
            end.record(self.stream)
            torch.cuda.synchronize(self.device)
            if world > 1:
                torch.distributed.barrier()
            elapsed_ms = start.elapsed_time(end)
            # keep the GPU busy (untimed) so that the clock sampler sees at least ~1.5 s of load
            g = self.g_main or self.g_rem
            while time.time() - t_wall < 1.5:
                g.replay()
                torch.cuda.synchronize(self.device)
        return elapsed_ms, clocks.summary()

    def bytes_per_launch(self):
        """Mean algorithmic and dense bytes of the captured steps (outputs read back)."""
        w, rows = self.w, self.w["per_step_rows"]
        n = self.chunk if self.reps else self.rem
        counts = self.out_c[:n].cpu().numpy()
        if not (counts >= 1).all():  # the synthetic workloads hold no invalid rows
            raise RuntimeError(f"{int((counts < 1).sum())} rows of the timed steps are not valid")
        alg, dense = [], []
        for s in range(n):
            r = (s % self.n_inputs) * rows
            if self.tree:
                sub = {k: (v[r:r + rows] if isinstance(v, np.ndarray) and v.shape[:1] == (w["target"].shape[0],)
                           else v) for k, v in w.items()}
                alg.append(algorithmic_bytes_tree(sub, counts[s], self.out_p[s].cpu().numpy()))
                dense.append(dense_bytes_tree(sub))
            else:
                b = algorithmic_bytes_chain(w, range(r, r + rows), counts[s])
                if self.sample:  # every draft row is read once more to draw the proposals
                    b += rows * w["tokens"].shape[1] * w["draft"].shape[2] * w["draft"].dtype.itemsize
                alg.append(b)
                dense.append(dense_bytes_chain(w, range(r, r + rows)))
        return float(np.mean(alg)), float(np.mean(dense)), float(counts.mean())

    def acceptance(self, max_sets=64):
        """Per-position acceptance, untimed, for chain workloads with sampling rows: one
        verify call per input set (at most max_sets) asking for min(1, p_k(x_k)/q_k(x_k)).
        Its mean over the sampling rows that reached position k estimates
        alpha_k = sum_x min(p_k(x), q_k(x)), the expected acceptance of a token drawn
        from q_k; positions after a row's first rejection are not evaluated (-1)."""
        import torch
        import speculative_decoding_verification_53_gb300 as sv
        if self._chain_inputs is None:
            return None
        dt, dd, dtok, dtemp, kind, seed = self._chain_inputs
        rows = self.w["per_step_rows"]
        sampling = torch.from_numpy(np.asarray(self.w["temperature"]) > 0)
        if not bool(sampling.any()):
            return None
        probs, keep = [], []
        with torch.cuda.stream(self.stream):
            for i in range(min(self.n_inputs, max_sets)):
                sl = slice(i * rows, (i + 1) * rows)
                _, _, ap = sv.spec_verify_chain(dt[sl], dd[sl], dtok[sl], dtemp[sl], seed, i, draft_kind=kind,
                                                want_accept_prob=True)
                probs.append(ap)
                keep.append(sampling[sl])
        torch.cuda.synchronize(self.device)
        ap = torch.cat(probs).cpu().numpy()
        on = torch.cat(keep).numpy()[:, None] & (ap >= 0)
        n = on.sum(0)
        alpha = [float(ap[on[:, k], k].mean()) if n[k] else None for k in range(ap.shape[1])]
        return {"alpha_per_position": alpha, "rows_per_position": [int(x) for x in n],
                "estimate": "mean of min(1, p_k(x_k)/q_k(x_k)) over the sampling rows that reached position k "
                            "(the library's out_accept_prob, one untimed call per input set)"}



def l2_note(w):
    """How the timed region avoids L2 reuse of inputs, from the workload's shapes."""
    rows = w["per_step_rows"]
    n_inputs = w["target"].shape[0] // rows
    set_mb = (w["target"].nbytes + w["draft"].nbytes) / n_inputs / 1e6
    if n_inputs > 1:
        return (f"L2 flushed ({L2_FLUSH_BYTES >> 20} MB read) right before the timed region; "
                f"{n_inputs} resident input sets of {set_mb:.1f} MB cycled, so no set is read twice within "
                f"{n_inputs * set_mb:.0f} MB of other inputs")
    return (f"L2 flushed ({L2_FLUSH_BYTES >> 20} MB read) right before the timed region; one resident input set "
            f"of {set_mb:.0f} MB, larger than L2, read every step")


def roofline_entry(bytes_per_launch, dense_bytes, ms_per_step, traffic, prof, kernel):
    peak, peak_src = measured_peak()
    achieved = bytes_per_launch / (ms_per_step / 1e3) / 1e9
    dense = dense_bytes / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs (STREAM copy)",
            "algorithmic_bytes_per_launch": bytes_per_launch,
            "algorithmic_bytes": "rows the rule reads: target rows up to the first rejection (tree: the visited "
                                 "nodes), the draft rows evaluated there, gathered draft entries, outputs",
            "dense_bytes_per_launch": dense_bytes, "dense_achieved": dense, "dense_frac": dense / peak,
            "dense_bytes": "every row of the call: all target rows, plus every draft-logit row of sampling rows "
                           "(draft probabilities: the gathered entries and one row)",
            "kernel": kernel, "traffic_source": prof}


# workloads reported beside the headline in the default line: (key, make_workload name,
# temperature); the large batch shares one set of logits across its temperatures
SIDE_WORKLOADS = [("large_batch_T0.7", "large_batch", 0.7), ("large_batch_T0", "large_batch", 0.0),
                  ("large_batch_T1.5", "large_batch", 1.5), ("mixed_batch", "mixed_batch", None),
                  ("tree", "tree", None)]


def run_side_workloads(args, rank, world, device, stream):
    """The other verify workloads, each timed like the headline (same steps, warm-up, L2
    flush) with its roofline and the oracle's bounded CPU baseline."""
    import torch
    out = {}
    large, large_dev = None, None
    gpu = device.index if device.index is not None else 0
    for key, name, T in SIDE_WORKLOADS:
        if name == "large_batch":
            if large is None:
                large = make_workload("large_batch", rank, args.rounds, 0, 0.7)
                large_dev = {k: to_dev(large[k], device) for k in ("target", "draft")}
            w = large if T == 0.7 else dict(large_batch_at(large, T), desc=large["desc"].replace("T=0.7", f"T={T:g}"))
            dev_inputs = large_dev
        else:
            w = make_workload(name, rank, args.rounds)
            dev_inputs = None
        t = Timed(w, device, stream, args.steps, args.warmup, dev_inputs=dev_inputs)
        elapsed, clocks = t.run(world, gpu)
        max_ms = slowest_rank_ms(elapsed, world, device)
        ms = max_ms / args.steps
        alg, dense, mean_count = t.bytes_per_launch()
        # the large batch at another temperature has its own summary (large_batch_T0, large_batch_T1.5)
        traffic, prof, pk = profile_traffic(key if name == "large_batch" and T != 0.7 else name)
        entry = {"workload": w["desc"], "ms_per_step": ms,
                 "value": whole_job_rate(w["per_step_rows"], args.steps, world, max_ms),
                 "unit": "trees/s" if w["kind"] == "tree" else UNIT, "mean_tokens_per_round": mean_count,
                 "l2": l2_note(w), "clocks": clocks,
                 "roofline": roofline_entry(alg, dense, ms, traffic, prof, pk or "kernel chosen by the library")}
        acc = t.acceptance()
        if acc is not None:
            entry["acceptance"] = acc
        if rank == 0 and not args.no_cpu_baseline:
            entry["cpu_baseline"] = run_cpu_baseline(w, w["per_step_rows"], t.n_inputs, w["kind"] == "tree",
                                                     budget_s=4.0)
        out[key] = entry
        del t
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, device):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    from speculative_decoding_verification_53_gb300 import build as svbuild

    if rank == 0:
        svbuild.build()
    if world > 1:
        torch.distributed.barrier()
    sv.lib()
    w = make_workload(args.workload, rank, args.rounds, args.batch, args.temperature)
    tree = w["kind"] == "tree"
    per_step_rows = w["per_step_rows"]
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    t = Timed(w, device, stream, args.steps, args.warmup)
    elapsed_ms, clock = t.run(world, device.index if device.index is not None else 0)
    bytes_per_launch, dense_bytes, mean_count = t.bytes_per_launch()
    acceptance = t.acceptance()
    n_inputs, resident = t.n_inputs, t.resident_bytes
    del t

    max_ms = slowest_rank_ms(elapsed_ms, world, device)
    ms_per_step = max_ms / args.steps
    value = whole_job_rate(per_step_rows, args.steps, world, max_ms)

    # end to end: host buffers, copies inside the timed region, through the public API
    kind = "probs" if w["draft_kind"] == 0 else "logits"
    e2e = run_e2e(args, w, device, stream, tree, per_step_rows, n_inputs, kind)

    cpu = run_cpu_baseline(w, per_step_rows, n_inputs, tree) if (rank == 0 and not args.no_cpu_baseline) else None
    side = None
    if args.workload == "single_stream" and not args.no_side_workloads:
        side = run_side_workloads(args, rank, world, device, stream)
    if rank != 0:
        return None
    prof_name = args.workload
    if args.workload == "large_batch" and args.temperature is not None and args.temperature != 0.7:
        prof_name = f"large_batch_T{args.temperature:g}"
    traffic, prof, prof_kernel = profile_traffic(prof_name, default_size=not (args.batch or args.rounds != 64 or (
        args.temperature is not None and args.workload != "large_batch")))
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, world),
        "resident_input_sets": n_inputs,
        "resident_bytes": resident,
        "mean_tokens_per_round": mean_count,
        "acceptance": acceptance,
        "roofline": roofline_entry(bytes_per_launch, dense_bytes, ms_per_step, traffic, prof,
                                   prof_kernel or ("tree_kernel" if tree else "chain kernel chosen by the library")),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": args.steps * (2 if w.get("sample") else 1),  # sampling + verify kernels per step
        "clocks": clock,
    }
    if side is not None:
        line["workloads"] = side
    return line


def workload_config(w, world):
    """The `config` object of both arms: the workload, its batch rows per step, how it
    is timed and how it is parallelised."""
    return {"workload": w["desc"], "batch_rows_per_step": w["per_step_rows"], "l2": l2_note(w),
            "timing": "CUDA-graph replay, CUDA events on the launching stream",
            "parallelism": f"replicas x{world}"}


def _packed(arrays, device, copies=1):
    """One pinned host buffer holding the arrays back to back (16-byte aligned offsets),
    `copies` device buffers of the same size, and device views of each array in each."""
    import torch
    parts, off = [], 0
    for a in arrays:
        a = np.ascontiguousarray(a)
        parts.append((off, a))
        off += (a.nbytes + 15) // 16 * 16
    host = torch.zeros(off, dtype=torch.uint8).pin_memory()
    hv = host.numpy()
    for o, a in parts:
        hv[o:o + a.nbytes] = np.frombuffer(a.tobytes(), dtype=np.uint8)
    devs, views = [], []
    for _ in range(copies):
        dev = torch.empty(off, dtype=torch.uint8, device=device)
        v = []
        for o, a in parts:
            dt = torch.bfloat16 if a.dtype == np.uint16 else getattr(torch, a.dtype.name)
            v.append(dev[o:o + a.nbytes].view(dt).view(a.shape))
        devs.append(dev)
        views.append(v)
    return host, devs, views


def _run_e2e_chain_host(w, device, stream, rows, n, kind):
    """The chain's round trip through spec_verify_chain_host (the C entry that takes host
    buffers): every step one copy of the packed inputs in, the verify, one copy of the
    tokens and counts out.  E2E_STREAMS streams take the steps in turn, each with its own
    device buffers and workspace, so a step's copy in overlaps the verifies (and the fixed
    start-up latency of the copies) of the steps before it, as a serving loop with several
    independent requests in flight would pipeline them.  The entry is called through ctypes
    with its arguments prepared once, so the host does not pace the loop."""
    import ctypes
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    sl = slice(0, rows)
    K, V = w["tokens"].shape[1], w["target"].shape[2]
    tdt = torch.bfloat16 if w["target"].dtype == np.uint16 else torch.float32
    ddt = torch.bfloat16 if w["draft"].dtype == np.uint16 else torch.float32
    offs, nin, nout = sv.spec_verify_host_sizes(rows, K, V, target_dtype=tdt, draft_dtype=ddt, draft_kind=kind)
    hin = torch.zeros(nin, dtype=torch.uint8).pin_memory()
    hv = hin.numpy()
    for o, k in zip(offs, ("target", "draft", "tokens", "temperature")):
        a = np.ascontiguousarray(w[k][sl])
        hv[o:o + a.nbytes] = np.frombuffer(a.tobytes(), dtype=np.uint8)
    ns = E2E_STREAMS
    streams = [stream] + [torch.cuda.Stream(device) for _ in range(ns - 1)]
    dins = [torch.empty(nin, dtype=torch.uint8, device=device) for _ in range(ns)]
    douts = [torch.empty(nout, dtype=torch.uint8, device=device) for _ in range(ns)]
    houts = [torch.zeros(nout, dtype=torch.uint8).pin_memory() for _ in range(ns)]
    ws_bytes = max(sv.spec_verify_workspace_size(rows, K, V), 256)
    wss = [torch.zeros(ws_bytes, dtype=torch.uint8, device=device) for _ in range(ns)]
    fn = sv.lib().spec_verify_chain_host
    vp = ctypes.c_void_p
    codes = (sv.SV_BF16 if tdt == torch.bfloat16 else sv.SV_F32, sv.SV_BF16 if ddt == torch.bfloat16 else sv.SV_F32,
             sv.SV_DRAFT_PROBS if kind == "probs" else sv.SV_DRAFT_LOGITS)
    per = [(vp(hin.data_ptr()), vp(dins[j].data_ptr()), vp(houts[j].data_ptr()), vp(douts[j].data_ptr()))
           + codes + (rows, K, V) for j in range(ns)]
    tail = [(vp(wss[j].data_ptr()), ws_bytes, vp(streams[j].cuda_stream)) for j in range(ns)]

    def one(i):
        j = i % ns
        st = fn(*per[j], 23, i, *tail[j])
        if st != sv.SV_OK:
            raise sv.SpecVerifyError(st, "spec_verify_chain_host")

    for i in range(2 * ns):
        one(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(streams[0])
    for s in streams[1:]:
        s.wait_event(start)
    for i in range(n):
        one(i)
    for s in streams[1:]:
        done = torch.cuda.Event()
        done.record(s)
        streams[0].wait_event(done)
    end.record(streams[0])
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    for j in range(ns):  # the device copy holds the inputs, and every row of the last steps verified
        if not torch.equal(dins[j].cpu(), hin):
            raise RuntimeError("end-to-end staging of the inputs is wrong")
        counts = houts[j].view(torch.int32)[rows * (K + 1):]
        if not (counts >= 1).all():
            raise RuntimeError("end-to-end counts are not all valid")
    return {"value": rows * n / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(nin),
            "d2h_bytes_per_step": int(nout), "steps": n, "ms_per_step": ms / n,
            "staging": "spec_verify_chain_host: inputs packed in one pinned buffer (one copy in), tokens and counts "
                       f"in one (one copy out); {ns} streams take the steps in turn, so a step's copy in overlaps "
                       "the verifies of the steps before it"}


def run_e2e(args, w, device, stream, tree, per_step_rows, n_inputs, kind):
    """Through the public API with host buffers, every step: the step's inputs copied from
    pinned host memory (staged back to back, one copy), the verify call (outputs and
    workspace preallocated, as a serving loop would), the tokens and counts copied back
    to pinned host memory (one copy).  No synchronisation inside the loop."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    n = min(args.e2e_steps, max(args.steps, 3))
    sl = slice(0, per_step_rows)
    if tree:
        names = ["target", "draft", "node_tokens", "parent", "temperature"]
        D = w["max_depth"]
        out_cols = D + 1
    elif w.get("sample"):  # the drafted tokens are an output here
        names = ["target", "draft", "temperature"]
        out_cols = w["tokens"].shape[1] + 1
    else:
        names = ["target", "draft", "tokens", "temperature"]
        out_cols = w["tokens"].shape[1] + 1
    if not tree and not w.get("sample"):
        return _run_e2e_chain_host(w, device, stream, per_step_rows, n, kind)
    hin, dins, vs = _packed([w[k][sl] for k in names], device)
    din, views = dins[0], vs[0]
    # outputs back to back in one device buffer: tokens [B][cols], count [B] (and the
    # tree's path, not read back)
    dout = torch.empty(per_step_rows * (out_cols + 1), dtype=torch.int32, device=device)
    ot = dout[:per_step_rows * out_cols].view(per_step_rows, out_cols)
    oc = dout[per_step_rows * out_cols:]
    hout = torch.empty_like(dout, device="cpu").pin_memory()
    opath = torch.empty((per_step_rows, D), dtype=torch.int32, device=device) if tree else None
    odraft = torch.empty((per_step_rows, w["tokens"].shape[1]), dtype=torch.int32, device=device) \
        if w.get("sample") else None
    K = w["tokens"].shape[1] if not tree else 0
    ws_bytes = sv.spec_verify_workspace_size(per_step_rows, K, w["target"].shape[2]) if not tree else 0
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=device) if not tree else None

    def one(i):
        din.copy_(hin, non_blocking=True)
        if tree:
            dt, dd, dtok, dpar, dtemp = views
            sv.spec_verify_tree(dt, dd, dtok, dpar, dtemp, D, 23, i, draft_kind=kind,
                                sibling_rule=w.get("sibling_rule", "without_replacement"),
                                out_tokens=ot, out_count=oc, out_path=opath)
        elif w.get("sample"):
            dt, dd, dtemp = views
            sv.spec_sample_and_verify(dt, dd, dtemp, 23, i, out_draft_tokens=odraft, out_tokens=ot, out_count=oc,
                                      workspace=ws)
        else:
            dt, dd, dtok, dtemp = views
            sv.spec_verify_chain(dt, dd, dtok, dtemp, 23, i, draft_kind=kind, out_tokens=ot, out_count=oc,
                                 workspace=ws)
        hout.copy_(dout, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(n):
        one(i)
    end.record(stream)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    for k, v in zip(names, views):  # the staged views hold exactly the step's inputs
        a = np.ascontiguousarray(w[k][sl])
        got = v.cpu().view(torch.int16).numpy().view(np.uint16) if a.dtype == np.uint16 else v.cpu().numpy()
        if not np.array_equal(got.view(np.uint8), a.view(np.uint8)):
            raise RuntimeError(f"end-to-end staging of {k} is wrong")
    if not (hout[per_step_rows * out_cols:] >= 1).all():  # every row of the last step verified
        raise RuntimeError("end-to-end counts are not all valid")
    return {"value": per_step_rows * n / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(hin.numel()),
            "d2h_bytes_per_step": int(hout.numel() * 4), "steps": n, "ms_per_step": ms / n,
            "staging": "inputs packed in one pinned buffer (one copy in), tokens and counts in one (one copy out)"}


def run_cpu_baseline(w, per_step_rows, n_inputs, tree, budget_s=10.0):
    """The oracle (fp64, one thread, unmodified) on a bounded sample of the same workload."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    done = 0
    i = 0
    while time.perf_counter() - t0 < budget_s:
        r = (i % n_inputs) * per_step_rows
        sl = slice(r, r + per_step_rows)
        if tree:
            oracle.verify_tree(w["target"][sl], w["draft"][sl], w["node_tokens"][sl], w["parent"][sl],
                               w["temperature"][sl], w["max_depth"], 17, i, draft_kind=w["draft_kind"],
                               sibling_rule=1 if w.get("sibling_rule") == "iid" else 0)
        else:
            if w.get("sample"):
                oracle.sample_and_verify(w["target"][sl], w["draft"][sl], w["temperature"][sl], 17, i)
            else:
                oracle.verify_chain(w["target"][sl], w["draft"][sl], w["tokens"][sl], w["temperature"][sl], 17, i,
                                    draft_kind=w["draft_kind"])
        done += per_step_rows
        i += 1
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{i} steps ({done} verify rows) of the same workload in {el:.1f} s, single thread, fp64"}


# ---------------------------------------------------------- reference arm

def run_reference(args, rank):
    """The oracle as it stands, timed on the host cores, on the same workload, metric and unit."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = make_workload(args.workload, 0, args.rounds, args.batch, args.temperature)
    per_step_rows = w["per_step_rows"]
    n_inputs = w["target"].shape[0] // per_step_rows
    tree = w["kind"] == "tree"
    budget = 120.0

    def one(i):
        r = (i % n_inputs) * per_step_rows
        sl = slice(r, r + per_step_rows)
        if tree:
            oracle.verify_tree(w["target"][sl], w["draft"][sl], w["node_tokens"][sl], w["parent"][sl],
                               w["temperature"][sl], w["max_depth"], 17, i, draft_kind=w["draft_kind"],
                               sibling_rule=1 if w.get("sibling_rule") == "iid" else 0)
        else:
            if w.get("sample"):
                oracle.sample_and_verify(w["target"][sl], w["draft"][sl], w["temperature"][sl], 17, i)
            else:
                oracle.verify_chain(w["target"][sl], w["draft"][sl], w["tokens"][sl], w["temperature"][sl], 17, i,
                                    draft_kind=w["draft_kind"])

    for i in range(max(args.warmup, 3)):
        one(i)
        if i >= 3 and args.warmup > 3:
            break
    t0 = time.perf_counter()
    done = 0
    while done < args.steps and (time.perf_counter() - t0) < budget:
        one(done)
        done += 1
    el = time.perf_counter() - t0
    value = done * per_step_rows / el
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": done,
            "warmup": max(args.warmup, 3), "ms_per_step": el / max(done, 1) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(w, args.gpus), "steps_requested": args.steps, "time_budget_s": budget,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{done} steps of the workload on one host core (fp64 C oracle)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------ steps around a tree verify

AUX_WORKLOADS = ("tree_mask", "kv_compact")
KV_LAYOUT = dict(n_buffers=64, heads=8, rows=1024, dim=128, nodes=60, depth=6, sets=16)


def make_aux(args, rank):
    from speculative_decoding_verification_53_gb300 import synth
    seed = 2000 + rank
    if args.workload == "tree_mask":
        B = args.batch or 1024
        N = args.nodes or 1024
        par = synth.random_parents(seed, B, N, shape="bfs", branch=3, max_depth=6 if N <= 64 else 16)
        W = (N + 31) // 32
        bytes_per_step = B * N * 4 + B * N * W * 4 + B * N * 4 + B * 4
        # distinct parent and output buffers per step, cycled, so that the bytes touched
        # between two uses of one buffer exceed twice the L2 (129 MB)
        n_sets = max(2, -(-2 * (129 << 20) // bytes_per_step))
        chunk = min(args.steps, 1000)
        n_graphs = -(-n_sets // chunk) if n_sets > chunk else 1
        n_sets = n_graphs * chunk if n_sets > chunk else n_sets
        return dict(parent=par, B=B, N=N, W=W, metric=f"tree-attention masks/s (N={N}-node draft trees)",
                    unit="trees/s", per_step=B, n_sets=n_sets, n_graphs=n_graphs,
                    l2="%d distinct parent/output sets cycled (%.0f MB between reuses, larger than L2)" % (
                        n_sets, n_sets * bytes_per_step / 1e6),
                    bytes_per_step=bytes_per_step,
                    desc=f"tree-attention mask, B={B} trees of N={N} nodes (breadth-first, up to 3 children, "
                         f"depth<={6 if N <= 64 else 16}), uint32 ancestor bitmask [B][N][{W}] + depth")
    L = dict(KV_LAYOUT)
    B = args.batch or 32
    par = synth.random_parents(seed, B * L["sets"], L["nodes"], max_depth=L["depth"])
    path, count = synth.accepted_paths(seed, par, L["depth"])
    base = np.repeat(np.arange(L["sets"], dtype=np.int32) * (L["rows"] // L["sets"]), B)
    moves = np.array([sum(1 for d in range(c - 1) if p[d] != d) for p, c in zip(path, count)])
    row_bytes = L["dim"] * 2
    per_set = moves.reshape(L["sets"], B).sum(1) * 2 * row_bytes * L["heads"] * L["n_buffers"]
    return dict(path=path, count=count, base=base, B=B, layout=L, per_step=B,
                l2=f"{L['sets']} path sets in disjoint cache windows cycled (touched bytes per cycle > L2)",
                metric="accepted-path KV compactions/s (batch rows, every layer's K and V)", unit="batch rows/s",
                bytes_per_set=per_set, row_bytes=row_bytes,
                desc=f"accepted-path KV compaction, B={B}, {L['n_buffers']} cache tensors (32 layers x K,V) of "
                     f"[B][{L['heads']} heads][{L['rows']} rows][{L['dim']}] bf16, tree of {L['nodes']} nodes, "
                     f"depth<={L['depth']}, {L['sets']} resident path sets in disjoint row windows")


def aux_config(a, world):
    """The `config` object of both arms for the steps around a tree verify."""
    return {"workload": a["desc"], "batch_rows_per_step": a["per_step"], "l2": a["l2"],
            "timing": "CUDA-graph replay, CUDA events on the launching stream", "parallelism": f"replicas x{world}"}


def run_aux(args, rank, world, device):
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    from speculative_decoding_verification_53_gb300 import build as svbuild
    if rank == 0:
        svbuild.build()
    if world > 1:
        torch.distributed.barrier()
    sv.lib()
    a = make_aux(args, rank)
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    chunk = min(args.steps, 1000)
    n_graphs = 1
    if args.workload == "tree_mask":
        n_sets, n_graphs = a["n_sets"], a["n_graphs"]
        dpar = torch.from_numpy(a["parent"]).to(device).unsqueeze(0).repeat(n_sets, 1, 1)
        om = torch.empty((n_sets, a["B"], a["N"], a["W"]), dtype=torch.int32, device=device)
        od = torch.empty((n_sets, a["B"], a["N"]), dtype=torch.int32, device=device)
        ov = torch.empty((n_sets, a["B"]), dtype=torch.int32, device=device)

        def step(i):
            s = i % n_sets
            sv.spec_tree_mask(dpar[s], out_mask=om[s], out_depth=od[s], out_valid=ov[s])

        def bytes_of(i):
            return a["bytes_per_step"]
        kernel = "tree_mask_kernel"
    else:
        L = a["layout"]
        kv = torch.empty((L["n_buffers"], a["B"], L["heads"], L["rows"], L["dim"]), dtype=torch.bfloat16,
                         device=device)
        kv.fill_(1.0)
        bufs = [kv[k] for k in range(L["n_buffers"])]
        a["bufs"] = bufs
        dpath = torch.from_numpy(a["path"]).to(device)
        dcount = torch.from_numpy(a["count"]).to(device)
        dbase = torch.from_numpy(a["base"]).to(device)
        B = a["B"]

        def step(i):
            s = i % L["sets"]
            sl = slice(s * B, (s + 1) * B)
            sv.spec_kv_compact(bufs, dpath[sl], dcount[sl], dbase[sl])

        def bytes_of(i):
            return float(a["bytes_per_set"][i % L["sets"]])
        kernel = "kv_compact_kernel"

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(device)
    reps, rem = divmod(args.steps, chunk)
    graphs = []
    for j, n in enumerate([chunk] * (min(reps, n_graphs) if reps else 0) + ([rem] if rem else [])):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(j * chunk + i)
        graphs.append((g, n))
    full = graphs[:min(reps, n_graphs)] if reps else []
    for g, _ in graphs:
        g.replay()
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        t_wall = time.time()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        start.record(stream)
        for r in range(reps):
            full[r % len(full)][0].replay()
        if rem:
            graphs[-1][0].replay()
        end.record(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        elapsed_ms = start.elapsed_time(end)
        while time.time() - t_wall < 1.5:
            graphs[0][0].replay()
            torch.cuda.synchronize(device)
    clock = clocks.summary()
    max_ms = slowest_rank_ms(elapsed_ms, world, device)
    ms_per_step = max_ms / args.steps
    value = whole_job_rate(a["per_step"], args.steps, world, max_ms)
    bytes_per_launch = float(np.mean([bytes_of(i) for i in range(chunk)]))
    e2e = run_aux_e2e(args, a, device, stream)
    cpu = run_aux_cpu(args, a, budget_s=10.0) if (rank == 0 and not args.no_cpu_baseline) else None
    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    achieved = bytes_per_launch / (ms_per_step / 1e3) / 1e9
    traffic, prof, prof_kernel = profile_traffic(args.workload, default_size=not (args.batch or args.nodes))
    return {
        "metric": a["metric"], "value": value, "unit": a["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32" if args.workload == "tree_mask" else "u8", "data": "synthetic",
        "config": aux_config(a, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs (STREAM copy)",
                     "algorithmic_bytes_per_launch": bytes_per_launch, "kernel": prof_kernel or kernel,
                     "traffic_source": prof},
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps, "clocks": clock,
    }


def run_aux_e2e(args, a, device, stream):
    """Through the public API with host buffers: the inputs copied in and the result
    read back every step (the mask and depths; for the compaction the counts, the cache
    itself being device state)."""
    import torch
    import speculative_decoding_verification_53_gb300 as sv
    n = min(args.e2e_steps, max(args.steps, 3))
    if args.workload == "tree_mask":
        hpar = torch.from_numpy(a["parent"]).pin_memory()
        dpar = torch.empty_like(hpar, device=device)
        hm = torch.empty((a["B"], a["N"], a["W"]), dtype=torch.int32).pin_memory()
        hd = torch.empty((a["B"], a["N"]), dtype=torch.int32).pin_memory()
        h2d, d2h = hpar.numel() * 4, hm.numel() * 4 + hd.numel() * 4

        def one(i):
            dpar.copy_(hpar, non_blocking=True)
            m, d, _ = sv.spec_tree_mask(dpar)
            hm.copy_(m, non_blocking=True)
            hd.copy_(d, non_blocking=True)
    else:
        B = a["B"]
        bufs = a["bufs"]
        hp = torch.from_numpy(a["path"][:B]).pin_memory()
        hc = torch.from_numpy(a["count"][:B]).pin_memory()
        hb = torch.from_numpy(a["base"][:B]).pin_memory()
        dp, dc, db = (torch.empty_like(x, device=device) for x in (hp, hc, hb))
        ho = torch.empty_like(hc).pin_memory()
        h2d, d2h = (hp.numel() + hc.numel() + hb.numel()) * 4, ho.numel() * 4

        def one(i):
            dp.copy_(hp, non_blocking=True)
            dc.copy_(hc, non_blocking=True)
            db.copy_(hb, non_blocking=True)
            sv.spec_kv_compact(bufs, dp, dc, db)
            ho.copy_(dc, non_blocking=True)
    for i in range(3):
        one(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(n):
        one(i)
    end.record(stream)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    return {"value": a["per_step"] * n / (ms / 1e3), "unit": a["unit"], "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": ms / n}


def _aux_oracle_loop(a, workload, budget_s, max_steps=None):
    """Runs the oracle on successive steps of the workload until the budget (or
    max_steps) is spent; returns (steps, units, seconds, sample text)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    steps = units = 0
    if workload == "tree_mask":
        while time.perf_counter() - t0 < budget_s and (max_steps is None or steps < max_steps):
            oracle.tree_mask(a["parent"])
            steps += 1
            units += a["B"]
        return steps, units, time.perf_counter() - t0, f"{steps} full steps ({units} trees)"
    L = a["layout"]
    B = a["B"]
    # one cache tensor at a time: [B*heads][rows][row_bytes], compacted in place
    cache = np.zeros((B * L["heads"], L["rows"], a["row_bytes"]), np.uint8)
    t0 = time.perf_counter()
    tensors = 0
    while time.perf_counter() - t0 < budget_s and (max_steps is None or steps < max_steps):
        s = (tensors // L["n_buffers"]) % L["sets"]
        sl = slice(s * B, (s + 1) * B)
        oracle.kv_compact(cache, np.repeat(a["path"][sl], L["heads"], axis=0), np.repeat(a["count"][sl], L["heads"]),
                          np.repeat(a["base"][sl], L["heads"]), inplace=True)
        tensors += 1
        if tensors % L["n_buffers"] == 0:
            steps += 1
    el = time.perf_counter() - t0
    units = B * tensors / L["n_buffers"]
    return steps, units, el, f"{tensors} cache tensors ({tensors / L['n_buffers']:.1f} steps)"


def run_aux_cpu(args, a, budget_s=10.0):
    steps, units, el, sample = _aux_oracle_loop(a, args.workload, budget_s)
    return {"value": units / el, "unit": a["unit"], "cores": 1, "kind": "oracle",
            "sample": f"{sample} of the same workload in {el:.1f} s, single thread"}


def run_aux_reference(args, rank):
    if rank != 0:
        return None
    a = make_aux(args, 0)
    steps, units, el, sample = _aux_oracle_loop(a, args.workload, 120.0, max_steps=args.steps)
    value = units / el
    return {"metric": a["metric"], "value": value, "unit": a["unit"], "n_gpus": args.gpus, "steps": steps,
            "warmup": max(args.warmup, 3), "ms_per_step": el / max(steps, 1) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u32" if args.workload == "tree_mask" else "u8",
            "data": "synthetic", "impl": "reference",
            "config": aux_config(a, args.gpus), "steps_requested": args.steps, "time_budget_s": 120.0,
            "cpu_baseline": {"value": value, "unit": a["unit"], "cores": 1, "kind": "oracle",
                             "sample": f"{sample} on one host core (C oracle)"},
            "e2e": {"value": value, "unit": a["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# -------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="single_stream",
                    choices=["single_stream", "large_batch", "mixed_batch", "sample_verify", "tree", "tree_iid",
                             "tree_mask", "kv_compact"])
    ap.add_argument("--rounds", type=int, default=64, help="resident rounds of the single-stream workload")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--batch", type=int, default=0,
                    help="batch rows (large_batch: 256, tree_mask: 1024 trees, kv_compact: 32)")
    ap.add_argument("--nodes", type=int, default=0, help="tree nodes of the tree_mask workload (default 1024)")
    ap.add_argument("--temperature", type=float, default=None, help="temperature of the large-batch workload")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="default workload only: skip the large-batch, mixed-batch and tree entries of `workloads`")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    aux = args.workload in AUX_WORKLOADS
    if args.impl == "reference":
        line = run_aux_reference(args, rank) if aux else run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    line = run_aux(args, rank, world, device) if aux else run_ours(args, rank, world, device)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
