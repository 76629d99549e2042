#!/usr/bin/env python
"""Throughput of the speculative-decoding verification step on GB300.

One step = one verify call over one batch of the workload: B=256 requests,
K=5 one-hot draft positions, V=152064 bf16 logits (Qwen vocabulary), T=1.
The default prints one JSON line with calls/s (device-timed, inputs resident
in HBM), the roofline of the dominant kernel (logit bytes / kernel time
against the measured HBM copy bandwidth), an end-to-end figure through the
C ABI with host buffers, and the fp64 CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I]
  python bench.py --impl reference ...   (the oracle as the reference arm)

Multi-GPU (torchrun, one rank per GPU): every rank verifies its own batch
(weak scaling, no collective on the data path); timing is bracketed by
barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

METRIC = "verify calls/s and logits HBM GB/s (% of GB300 peak) at B=256 K=5 V=152064"
FALLBACK_HBM_GBS = 6800.0
# the sources of each profiled kernel (a profile's DRAM figure counts only
# while these are unchanged)
KERNEL_SOURCES = {
    "stream": ["token_verification_gb300/csrc/sv_stream.cuh",
               "token_verification_gb300/csrc/sv_verify.cu",
               "token_verification_gb300/csrc/sv_rows.cuh",
               "token_verification_gb300/csrc/sv_common.cuh"],
    "filter": ["token_verification_gb300/csrc/sv_filter.cu",
               "token_verification_gb300/csrc/sv_rows.cuh",
               "token_verification_gb300/csrc/sv_common.cuh"],
}


# ---------------------------------------------------------------------------
# distributed helpers (host logic; tested with gloo on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(base_seed, rank):
    """Each rank verifies its own batch (weak scaling): seed offset by rank."""
    return base_seed + 1000 * rank


def aggregate(elapsed_s, units, world, backend_device=None):
    """(max elapsed over ranks, total units over ranks); identity when world = 1."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=backend_device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------
# peaks, clocks, profile traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text):
    """C++ source without its // comments and blank runs: edits to comments
    alone do not change the compiled kernel."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0 and line.count('"', 0, i) % 2 == 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_source_hash(kind="stream"):
    """Hash of the code (comments left out) of the sources a profiled kernel
    is built from."""
    if kind not in KERNEL_SOURCES:
        return None
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic(name):
    """DRAM bytes per launch of the ncu capture `name` recorded in
    profiles/traffic.json, if it was taken on the current sources of its
    kernel (else None)."""
    if not name:
        return None
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[name]
    except (OSError, KeyError, ValueError):
        return None
    if entry.get("kernel_source_hash") != kernel_source_hash(entry.get("kernel", "")):
        return None
    return int(entry["dram_bytes_per_launch"])


# the ncu capture (profiles/traffic.json) of each benchmarked (workload, mode)
PROFILE_NAMES = {(2, "sample"): "verify_stream_onehot_B256_K5_V152064",
                 (7, "sample"): "filter_rows_topp_B256_K5_V152064"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (read-only)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self._stop = threading.Event()
        self._proc = None
        self._thread = None
        self.window = None

    def start(self):
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self._proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        if self.window:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            if inside:
                rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[1]) for _, p in rows if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in rows if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in rows:
            for name, val in zip(names, p[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# the CPU oracle baseline
# ---------------------------------------------------------------------------

def oracle_run(wl, mode, requests, threads):
    """Seconds the fp64 oracle takes on the first `requests` requests."""
    import oracle
    sub = slice(0, requests)
    t0 = time.perf_counter()
    if mode == "propose":
        oracle.ngram(wl.history[sub], wl.history_lens[sub], wl.meta["n_min"], wl.meta["n_max"],
                     wl.K)
    elif mode == "tree_typical":
        oracle.tree_typical(wl.target[sub], wl.parent, wl.node_tokens[sub], wl.uniforms[sub], wl.T,
                            wl.eps, wl.delta, wl.max_depth, threads=threads)
    elif mode == "typical":
        oracle.typical(wl.target[sub], wl.draft_tokens[sub], wl.uniforms[sub], wl.T, wl.eps,
                       wl.delta, threads=threads)
    elif mode == "tree":
        oracle.tree(wl.target[sub], wl.parent, wl.node_tokens[sub], wl.max_depth, threads=threads)
    elif mode == "tree_sample":
        oracle.tree_sample(wl.target[sub], wl.parent, wl.node_tokens[sub], wl.uniforms[sub], wl.T,
                           wl.max_depth, threads=threads)
    elif mode == "greedy":
        oracle.greedy(wl.target[sub], wl.draft_tokens[sub], threads=threads,
                      token_mask=None if wl.token_mask is None else wl.token_mask[sub])
    else:
        oracle.sample(wl.target[sub], None if wl.draft is None else wl.draft[sub],
                      wl.draft_tokens[sub], wl.uniforms[sub], wl.T, threads=threads,
                      token_mask=None if wl.token_mask is None else wl.token_mask[sub],
                      top_k=wl.top_k, top_p=float(np.float32(wl.top_p)))
    return time.perf_counter() - t0


def _oracle_rate(wl, mode, threads, budget_s):
    """Calls/s of the oracle with `threads` threads: the median of 3 timed
    runs over a sample of requests sized to about budget_s / 3 each."""
    probe = min(wl.B, max(threads, 2))
    per_req = oracle_run(wl, mode, probe, threads) / probe
    reqs = min(wl.B, max(probe, int(budget_s / 3 / max(per_req, 1e-9))))
    reps = max(1, min(200, int(budget_s / 3 / max(per_req * reqs, 1e-9)))) if reqs == wl.B else 1
    rates = []
    for _ in range(3):
        t = sum(oracle_run(wl, mode, reqs, threads) for _ in range(reps))
        rates.append((reps * reqs / wl.B) / t)
    return statistics.median(rates), "%d x %d of the B=%d requests, median of 3" % (reps, reqs, wl.B)


def cpu_baseline(wl, mode, budget_s=12.0):
    """The oracle on the host cores (all threads) and on one thread."""
    threads = os.cpu_count() or 1
    value, sample = _oracle_rate(wl, mode, threads, budget_s)
    single, s_sample = _oracle_rate(wl, mode, 1, budget_s / 3)
    return {"value": value, "unit": "calls/s", "cores": threads, "kind": "oracle",
            "sample": sample + " (%d threads)" % threads,
            "single_thread": {"value": single, "unit": "calls/s", "cores": 1,
                              "sample": s_sample}}


def load_workload(args, seed=0, index=None, greedy=None):
    from token_verification_gb300 import synth
    index = args.workload if index is None else index
    greedy = args.greedy if greedy is None else greedy
    wl = synth.make_workload(index, seed=seed)
    typical = wl.meta.get("typical", False)
    tree_kind = "tree_typical" if typical else (
        "tree_sample" if (wl.uniforms is not None and wl.uniforms.ndim == 2) else "tree")
    mode = ("propose" if wl.history is not None
            else tree_kind if wl.parent is not None
            else "greedy" if greedy else "typical" if typical else "sample")
    if args.batch:  # a smaller batch of the same workload (profiling captures)
        wl.B = args.batch
        for name in ("target", "draft", "draft_tokens", "uniforms", "node_tokens", "token_mask",
                     "history", "history_lens"):
            v = getattr(wl, name)
            if v is not None:
                setattr(wl, name, v[:args.batch])
        wl.meta["workload"] += "-first%d" % args.batch
    return wl, mode


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, each step one
    whole call (every request of the batch)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl, mode = load_workload(args)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_run(wl, mode, wl.B, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_run(wl, mode, wl.B, threads)
    value = args.steps / t
    line = {"impl": "reference", "metric": metric_name(wl, mode, args), "value": value,
            "unit": "calls/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, mode),
            "cpu_baseline": {"value": value, "unit": "calls/s", "cores": threads, "kind": "oracle",
                             "sample": "every step a whole call: all %d requests" % wl.B},
            "e2e": {"value": value, "unit": "calls/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def metric_name(wl, mode, args):
    if args.workload == 2 and mode == "sample" and not args.batch:
        return METRIC
    if mode == "propose":
        return "n-gram proposer calls/s and context GB/s on %s" % wl.meta["workload"]
    return "verify calls/s and logits HBM GB/s (%% of GB300 peak) on %s (%s)" % (
        wl.meta["workload"], mode)


L2_BYTES = 129 * 2**20  # GB300


def input_bytes(wl, mode):
    """Bytes of one input set (what a call reads from its inputs)."""
    if mode == "propose":
        return int(wl.history.nbytes)
    total = wl.target.nbytes
    if wl.draft is not None and mode == "sample":
        total += wl.draft.nbytes
    if wl.token_mask is not None:
        total += wl.token_mask.nbytes
    return int(total)


def n_input_sets(set_bytes):
    """Input sets to rotate through so that a set comes back only after more
    than twice the L2's capacity of other inputs: 2 when a set is larger
    than L2, else at least 4 (at most 4096)."""
    if set_bytes > L2_BYTES:
        return 2
    return int(min(4096, max(4, 1 + math.ceil(2 * L2_BYTES / max(set_bytes, 1)))))


def workload_config(wl, mode):
    cfg = {"workload": wl.meta["workload"], "mode": mode, "B": wl.B, "V": wl.V,
           "logits": wl.dtype, "parallelism": "dp%d" % dist_env()[0]}
    if mode == "propose":
        del cfg["logits"]
        cfg.update(L=wl.meta["L"], K=wl.K, n_min=wl.meta["n_min"], n_max=wl.meta["n_max"])
    elif mode in ("tree", "tree_typical", "tree_sample"):
        cfg.update(N=int(wl.parent.size), max_depth=wl.max_depth)
        if mode == "tree_typical":
            cfg.update(temperature=wl.T, eps=wl.eps, delta=wl.delta)
        if mode == "tree_sample":
            cfg.update(temperature=wl.T)
    else:
        cfg.update(K=wl.K, drafts=wl.meta.get("drafts"), temperature=0.0 if mode == "greedy" else wl.T)
        if wl.token_mask is not None:
            cfg["grammar_masks"] = dict(wl.meta["grammar"], bytes=int(wl.token_mask.nbytes))
        if mode == "sample" and (wl.top_k or wl.top_p < 1.0):
            cfg.update(top_k=wl.top_k, top_p=wl.top_p)
        if mode == "typical":
            cfg.update(eps=wl.eps, delta=wl.delta)
    nb, ns = input_bytes(wl, mode), n_input_sets(input_bytes(wl, mode))
    cfg["l2"] = ("%s: %d rotating input sets of %.1f MB (a set returns after %.0f MB of other "
                 "inputs, more than twice the %d MB L2)"
                 % ("inputs larger than L2" if nb > L2_BYTES else "inputs smaller than L2", ns,
                    nb / 2**20, (ns - 1) * nb / 2**20, L2_BYTES // 2**20))
    return cfg


class Case:
    """One workload resident on the device: `n_sets` input sets (copies,
    the requests rotated), enough that a set is not in L2 when it comes
    back, and the C-ABI call on them."""

    def __init__(self, wl, mode, device, n_sets=None):
        import torch
        from token_verification_gb300 import api
        self.api, self.torch = api, torch
        self.wl, self.mode, self.device = wl, mode, device
        to_t = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) \
            if wl.dtype == "bf16" else (lambda a: torch.from_numpy(a))
        self.host = {"target": to_t(wl.target)} if mode != "propose" else {
            "history": torch.from_numpy(wl.history),
            "history_lens": torch.from_numpy(wl.history_lens)}
        if mode == "propose":
            pass
        elif mode in ("tree", "tree_typical", "tree_sample"):
            self.host["node_tokens"] = torch.from_numpy(wl.node_tokens)
            self.host["parent"] = torch.from_numpy(np.ascontiguousarray(wl.parent, np.int32))
            if mode in ("tree_typical", "tree_sample"):
                self.host["uniforms"] = torch.from_numpy(wl.uniforms)
        else:
            self.host["tokens"] = torch.from_numpy(wl.draft_tokens)
            if wl.token_mask is not None:
                self.host["token_mask"] = torch.from_numpy(wl.token_mask.view(np.int32))
            if mode in ("sample", "typical"):
                self.host["uniforms"] = torch.from_numpy(wl.uniforms)
                if wl.draft is not None:
                    self.host["draft"] = to_t(wl.draft)
        B = wl.B
        self.n_sets = n_input_sets(input_bytes(wl, mode)) if n_sets is None else n_sets
        base = {k: v.to(device) for k, v in self.host.items()}
        self.sets = []
        for s in range(self.n_sets):
            perm = torch.from_numpy(np.roll(np.arange(B), (s * max(1, B // 2)) % max(B, 1))).to(device)
            self.sets.append({k: (v.clone() if k == "parent" else v[perm].contiguous())
                              for k, v in base.items()})
        del base

    def alloc(self, packed=True):
        if self.mode in ("tree", "tree_typical", "tree_sample", "propose"):
            return None
        return self.api.alloc_outputs(self.wl.B, self.wl.K, self.device, packed=packed,
                                      accept_prob=packed and self.mode == "sample",
                                      status=packed)

    def call(self, inputs, out):
        wl, api = self.wl, self.api
        if self.mode == "propose":
            return api.spec_ngram_propose(inputs["history"], inputs["history_lens"], K=wl.K,
                                          n_min=wl.meta["n_min"], n_max=wl.meta["n_max"], out=out)
        if self.mode == "tree":
            return api.spec_verify_tree(inputs["target"], inputs["parent"], inputs["node_tokens"],
                                        wl.max_depth, out, path=False, status=False)
        if self.mode == "tree_typical":
            return api.spec_verify_tree_typical(inputs["target"], inputs["parent"],
                                                inputs["node_tokens"], inputs["uniforms"], wl.T,
                                                wl.eps, wl.delta, wl.max_depth, out, path=False,
                                                status=False)
        if self.mode == "tree_sample":
            return api.spec_verify_tree_sample(inputs["target"], inputs["parent"],
                                               inputs["node_tokens"], inputs["uniforms"], wl.T,
                                               wl.max_depth, out, path=False, status=False)
        if self.mode == "typical":
            return api.spec_verify_typical(inputs["target"], inputs["tokens"], inputs["uniforms"],
                                           wl.T, wl.eps, wl.delta, out)
        if self.mode == "greedy":
            return api.spec_verify_greedy(inputs["target"], inputs["tokens"], out,
                                          token_mask=inputs.get("token_mask"))
        return api.spec_verify_sample(inputs["target"], inputs.get("draft"), inputs["tokens"],
                                      inputs["uniforms"], wl.T, out,
                                      token_mask=inputs.get("token_mask"), top_k=wl.top_k,
                                      top_p=wl.top_p)

    def step(self, i, out):
        return self.call(self.sets[i % self.n_sets], out)

    def results(self, out):
        """The call's per-request token rows and lengths (what a caller reads back)."""
        if self.mode == "propose":
            return out.drafts, out.draft_lens
        return out.tokens, out.accept_len

    def launches(self):
        if self.mode in ("tree", "propose"):
            return 1
        # stream, finalize (the residual draw and the packed output included)
        return 2

    def kernel_label(self):
        if self.mode == "propose":
            return "ngram_kernel"
        if self.mode == "tree":
            return "tree_kernel"
        if self.mode == "tree_typical":
            return "verify_stream_kernel + tree_typical_kernel"
        if self.mode == "tree_sample":
            return "verify_stream_kernel + tree_sample_kernel"
        if self.mode == "typical":
            return "verify_stream_kernel + finalize_kernel (typical)"
        masked = ", grammar-masked" if self.wl.token_mask is not None else ""
        if self.mode == "sample" and (self.wl.top_k or self.wl.top_p < 1.0):
            return "filter_rows_kernel + finalize_kernel (top-k/top-p%s)" % masked
        if self.mode == "sample" and self.wl.draft is not None:
            return "verify_stream_kernel + finalize_kernel (dense%s)" % masked
        return "verify_stream_kernel + finalize_kernel (%s%s)" % (
            "greedy" if self.mode == "greedy" else "one-hot", masked)

    def algorithmic_bytes(self, out):
        """Bytes the method needs per call: every needed logit once
        (sampling, greedy), plus the grammar mask words when masked; the
        rows on the accepted path (greedy tree); every candidate row (the
        tree calls that reduce all rows); every context token (proposer)."""
        wl = self.wl
        if self.mode == "propose":
            return int(wl.history_lens.astype(np.int64).sum()) * 4
        esz = 2 if wl.dtype == "bf16" else 4
        if self.mode == "tree":
            rows = int(out.accept_len.sum().item())
            return rows * wl.V * esz
        if self.mode in ("tree_typical", "tree_sample"):
            return wl.B * (wl.parent.size + 1) * wl.V * esz
        rows = wl.B * (wl.K + 1) + (wl.B * wl.K if (self.mode == "sample" and wl.draft is not None)
                                     else 0)
        masks = 0 if wl.token_mask is None else wl.token_mask.nbytes
        return rows * wl.V * esz + masks


class Replay:
    """The case's calls captured in CUDA graphs of `per_graph` complete calls
    each, call i on input set i % n_sets, enough graphs to go through every
    set; replays cycle through the graphs.  A serving loop captures its
    decode step the same way, so host-side launch work does not gate the
    device."""

    def __init__(self, case, per_graph, out, stream):
        import torch
        self.per_graph = per_graph
        side = torch.cuda.Stream(case.device)
        side.wait_stream(stream)
        self.graphs = []
        n_graphs = max(1, -(-case.n_sets // per_graph)) if case.n_sets > per_graph else 1
        with torch.cuda.stream(side):
            for i in range(3):  # this stream's workspace is set up outside the capture
                out = case.step(i, out) or out
            torch.cuda.synchronize()
            for g in range(n_graphs):
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=side):
                    for i in range(per_graph):
                        out = case.step(g * per_graph + i, out) or out
                self.graphs.append(graph)
        torch.cuda.synchronize()
        self.out = out
        self.next = 0

    def replay(self, calls):
        """Queue exactly `calls` calls (a multiple of per_graph)."""
        for _ in range(calls // self.per_graph):
            self.graphs[self.next].replay()
            self.next = (self.next + 1) % len(self.graphs)


def per_graph_for(steps, cap):
    """The largest graph size up to `cap` that divides `steps`."""
    return max(d for d in range(1, max(1, min(cap, steps)) + 1) if steps % d == 0)


def timed_seconds(torch, stream, fn):
    """Device time of the work `fn` queues on `stream` (CUDA events)."""
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3


def measure_config(args, index, greedy, device, calls=1000, warmup=10, oracle_budget=4.0):
    """One workload's row of the per-config record: calls/s over `calls`
    graph-replayed calls (rotating input sets), the roofline fraction of its
    algorithmic bytes, and the oracle on the host cores."""
    import torch
    wl, mode = load_workload(args, index=index, greedy=greedy)
    case = Case(wl, mode, device)
    out = case.alloc(packed=True)
    stream = torch.cuda.current_stream(device)
    for i in range(warmup):
        out = case.step(i, out) or out
    torch.cuda.synchronize()
    rep = Replay(case, 100, out, stream)
    rep.replay(100 * max(1, len(rep.graphs)))  # one pass over every set
    sec = timed_seconds(torch, stream, lambda: rep.replay(calls))
    out = rep.out
    value = calls / sec
    algo = case.algorithmic_bytes(out)
    peak, _ = hbm_peak()
    tok, lens = case.results(out)
    row = {"workload": wl.meta["workload"], "mode": mode, "calls_per_s": value,
           "us_per_call": 1e6 / value,
           "draft_tokens_per_s": (value * wl.B * wl.K if mode in ("sample", "greedy", "typical")
                                  else None),
           "algorithmic_bytes": algo, "hbm_gbs": algo * value / 1e9,
           "frac": algo * value / 1e9 / peak,
           ("mean_draft_len" if mode == "propose" else "mean_accept_len"):
               float(lens.float().mean().item()),
           "input_sets": case.n_sets, "calls_timed": calls, "kernel": case.kernel_label()}
    if not args.no_cpu_baseline:
        row["cpu_baseline"] = cpu_baseline(wl, mode, budget_s=oracle_budget)
    del rep, case, out
    torch.cuda.empty_cache()
    return row


# every standard workload (the five of the brief first, then the extensions)
PER_CONFIG = [(0, False), (1, False), (2, False), (3, False), (3, True), (4, False),
              (5, False), (6, False), (7, False), (8, False), (9, False), (10, False)]


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from token_verification_gb300 import _native
    _native.lib()

    wl, mode = load_workload(args, seed=shard_seed(0, rank))
    case = Case(wl, mode, device)
    out = case.alloc(packed=True)
    stream = torch.cuda.current_stream(device)

    for i in range(args.warmup):
        out = case.step(i, out) or out
    torch.cuda.synchronize()

    # Exactly K calls are timed, replayed from CUDA graphs of `per_graph`
    # complete calls each (--no-graph: one Python call per step).
    steps = args.steps
    replay = None
    if not args.no_graph:
        replay = Replay(case, per_graph_for(steps, args.graph_calls), out, stream)
        out = replay.out
        replay.replay(replay.per_graph * len(replay.graphs))
        torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    ev0.record(stream)
    if replay is not None:
        replay.replay(steps)
    else:
        for i in range(steps):
            case.step(i, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    if sampler:
        sampler.mark(w0, w1)
    max_elapsed, total_calls = aggregate(elapsed, steps, world, device)
    mean_len = float(case.results(out)[1].float().mean().item())
    algo_bytes = case.algorithmic_bytes(out)

    # The roofline: the call's average duration over a longer window of the
    # same replay (CUDA events on the launching stream), every call complete
    # (the dominant kernel and the small per-request one), so the fraction
    # is a lower bound for the dominant kernel alone.
    roof_calls = 0
    if replay is not None:
        roof = Replay(case, 100, out, stream)
        roof.replay(100 * len(roof.graphs))
        roof_calls = 100 * max(10, len(roof.graphs))
        call_s = timed_seconds(torch, stream, lambda: roof.replay(roof_calls)) / roof_calls
        del roof
    else:
        call_s = elapsed / steps
    if sampler:
        sampler.stop()

    # end to end through the C ABI with host buffers (pinned): H2D of the
    # step's inputs, the call, D2H of its results, every step
    e2e = None
    if rank == 0 and not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in case.host.items()}
        dev_in = {k: torch.empty_like(v, device=device) for k, v in pin.items()}
        out_tok, out_len = case.results(out)
        res_tok = torch.empty(tuple(out_tok.shape), dtype=torch.int32).pin_memory()
        res_len = torch.empty((wl.B,), dtype=torch.int32).pin_memory()
        e2e_steps = max(3, min(args.steps, args.e2e_steps))

        def e2e_step():
            for k in pin:
                dev_in[k].copy_(pin[k], non_blocking=True)
            case.call(dev_in, out)
            res_tok.copy_(out_tok, non_blocking=True)
            res_len.copy_(out_len, non_blocking=True)

        for _ in range(2):
            e2e_step()
        e2e_s = timed_seconds(torch, stream, lambda: [e2e_step() for _ in range(e2e_steps)])
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = res_tok.numel() * 4 + res_len.numel() * 4
        e2e = {"value": e2e_steps / e2e_s, "unit": "calls/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    if rank == 0:
        peak, peak_kind = hbm_peak()
        achieved = algo_bytes / call_s / 1e9
        value = total_calls / max_elapsed
        line = {
            "metric": metric_name(wl, mode, args), "value": value, "unit": "calls/s",
            "n_gpus": world,
            "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * max_elapsed / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl, mode),
            "draft_tokens_per_s": (value * wl.B * wl.K if mode in ("sample", "greedy", "typical")
                                   else None),
            "hbm_gbs": algo_bytes * value / 1e9,
            ("mean_draft_len" if mode == "propose" else "mean_accept_len"): mean_len,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "kernel": case.kernel_label(), "call_ms": call_s * 1e3,
                         "calls_timed": roof_calls or steps,
                         "algorithmic_bytes": algo_bytes,
                         "traffic": profiled_traffic(PROFILE_NAMES.get((args.workload, mode)))},
            "gpu_launches": steps * case.launches(),
            "launch": ("CUDA graphs of %d calls, replayed" % replay.per_graph) if replay
                      else "one Python call per step",
            "clocks": sampler.summary() if sampler else None,
            "e2e": e2e,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(wl, mode)
        if world == 1 and not args.no_per_config and args.workload == 2 and not args.batch:
            del case, out, replay
            torch.cuda.empty_cache()
            rows = {}
            for index, greedy in PER_CONFIG:
                key = "%d%s" % (index, "-greedy" if greedy else "")
                try:
                    rows[key] = measure_config(args, index, greedy, device)
                except Exception as e:  # a failure is reported, not hidden
                    rows[key] = {"error": "%s: %s" % (type(e).__name__, e)}
            line["per_config"] = rows
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config record of every standard workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first BATCH requests (small profiling cases)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every timed call from Python instead of replaying a CUDA graph")
    ap.add_argument("--graph-calls", type=int, default=100,
                    help="calls captured in the replayed CUDA graph")
    ap.add_argument("--greedy", action="store_true",
                    help="greedy verification (temperature 0) of the workload's drafts")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
