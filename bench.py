"""Benchmark of one verify step: ancestor masks -> tree attention (one layer) ->
acceptance walk, on synthetic inputs shaped like the workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-per-workload]

Prints ONE JSON line on rank 0. The headline workload is the 70B serving
layer (batch 64, context 32768, 31-node trees, 64/8 heads, vocabulary
128256), the largest configuration. ``value`` is verified tree nodes per
second (per attention layer) over all ranks, with inputs resident in HBM;
``e2e`` repeats the measurement through the public API from pinned host
buffers with the copies inside the timed region: the prefix KV cache is
device-resident state, and each step's inputs (queries, the tree's own K/V
rows scattered into their cache slots, tree, uniforms, lengths, page table,
both logits arrays) travel in one packed host-to-device copy, issued on a
side stream one step ahead; the outputs are read back every step. Between timed steps the inputs rotate over enough copies that the
working set exceeds L2. Per-kernel times are taken inside the step: a second
capture of the step graph carries timing events between its kernels.
``per_workload`` repeats the step measurement on the four other workloads.
``--impl reference`` times the fp64 CPU oracle on the host cores instead
(the reference arm).

Multi-GPU: the path does not shard; each rank runs an independent replica of
the workload (weak scaling) and the step time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_inputs  # noqa: E402
from synth.gen import algorithmic_bytes  # noqa: E402

DEFAULT_WORKLOAD = "serving_70b"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def workload_by_name(name):
    for i, w in enumerate(WORKLOADS):
        if w.name == name:
            return i, w
    raise SystemExit(f"unknown workload {name}; choose from {[w.name for w in WORKLOADS]}")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """(burst, sustained) bf16 TFLOP/s of the measured cuBLAS GEMM, and their kind."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_hash(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(workload, chunks=0):
    """DRAM bytes per launch from a committed ncu summary of the same workload
    and chunk setting (0: the library's choice), if the source of the kernel
    it captured has not changed since (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{workload}@{chunks}" if chunks else workload]
        if e.get("source_hash") == source_hash(e["source"]):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def walk_bytes(w, parent: np.ndarray, path: np.ndarray, accept_len: np.ndarray) -> int:
    """Logits bytes an exact acceptance walk must read: the target row of every
    node the walk visits (the root, then each accepted node) and the draft row
    of every visited node that has children (its children were tested).
    Computed from a finished walk (path, accept_len); rows of nodes the walk
    never reached are not needed."""
    total = 0
    for b in range(parent.shape[0]):
        kids = set(int(x) for x in parent[b, 1:])
        for j in path[b, : int(accept_len[b]) + 1]:
            total += w.V * 4 * (2 if int(j) in kids else 1)
    return total


def visited_nodes(accept_len: np.ndarray) -> int:
    """Nodes a finished walk visited: the root plus every accepted node."""
    return int(np.asarray(accept_len, np.int64).sum()) + int(np.asarray(accept_len).shape[0])


def aggregate(local_ms: float, local_units: float, world: int, reduce_max, reduce_sum):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    ms = reduce_max(local_ms)
    units = reduce_sum(local_units)
    return ms, units / (ms / 1e3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
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
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the oracle on the host cores
# ---------------------------------------------------------------------------

def _oracle_inputs(inp, bs):
    """q and logical float32 K/V of sequences ``bs`` for the oracle, regenerated
    from the generator's streams (only those sequences)."""
    from synth.gen import logical_kv, bf16_bits_to_f32
    w = inp.w
    T = inp.seq_lens[bs].astype(np.int64) + w.N
    Tcap = int(T.max())
    K = np.zeros((len(bs), Tcap, w.Hkv, w.D), np.float32)
    V = np.zeros_like(K)
    cvt = (lambda x: bf16_bits_to_f32(x)) if w.dtype == "bf16" else (lambda x: x)
    for n, b in enumerate(bs):
        for g in range(w.Hkv):
            k, v = logical_kv(w, inp.seed, int(b), g, int(T[n]))
            K[n, : T[n], g] = cvt(k)
            V[n, : T[n], g] = cvt(v)
    return cvt(inp.q[bs]), K, V


def time_oracle(inp, budget_s=15.0, max_steps=20, steps=None, warmup=0, threads=None):
    """Time the fp64 oracle for the whole verify step on the host cores.

    Attention is timed on a bounded sample: at most two sequences (their K/V
    regenerated alone), and within them as many (node, head) rows as fit the
    budget, scaled to all B*N*Hq rows. Masks and the acceptance walk run on
    the whole batch. Without ``steps``: as many steps as fit in ``budget_s``
    (at most ``max_steps``). With ``steps``: ``warmup`` untimed steps, then
    exactly ``steps`` timed ones. Returns (seconds per step, sample text, cores)."""
    import oracle
    w = inp.w
    cores = threads or len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    nseq = min(w.B, 2)
    bs = np.linspace(0, w.B - 1, nseq).astype(np.int64)
    q, K, V = _oracle_inputs(inp, bs)
    sl, par = inp.seq_lens[bs], inp.parent[bs]
    rows_all = w.B * w.N * w.Hq
    rows_pool = nseq * w.N * w.Hq
    t0 = time.perf_counter()
    oracle.tree_attn(q, K, V, sl, par, rows=np.array([[0, 0, 0]]))
    one = max(time.perf_counter() - t0, 1e-6)
    per_step_budget = budget_s / 2 if steps is None else budget_s / max(1, steps + warmup)
    nsel = rows_pool
    if one * rows_pool / cores > per_step_budget:
        nsel = max(cores, min(rows_pool, int(per_step_budget * cores / one)))
    sel = np.linspace(0, rows_pool - 1, nsel).astype(np.int64)
    rows = np.stack([sel // (w.N * w.Hq), (sel // w.Hq) % w.N, sel % w.Hq], 1)
    scale = rows_all / nsel

    def accept_part():
        oracle.tree_mask(inp.parent)
        oracle.spec_accept(inp.target, inp.draft, inp.tokens, inp.parent, inp.u_accept,
                           inp.u_bonus)

    for _ in range(warmup):
        oracle.tree_attn(q, K, V, sl, par, rows=rows)
        accept_part()
    fixed = steps
    steps = 0
    t_attn = t_acc = 0.0
    start = time.perf_counter()
    while ((fixed is not None and steps < fixed) or
           (fixed is None and steps < max_steps and
            (steps == 0 or time.perf_counter() - start < budget_s))):
        t0 = time.perf_counter()
        oracle.tree_attn(q, K, V, sl, par, rows=rows)
        t1 = time.perf_counter()
        accept_part()
        t2 = time.perf_counter()
        t_attn += (t1 - t0) * scale
        t_acc += t2 - t1
        steps += 1
    per_step = (t_attn + t_acc) / steps
    sample = ((f"{warmup} untimed + " if warmup else "")
              + f"{steps} timed verify step(s) of {w.name}; attention on {nsel} of "
              + f"{rows_all} (node, head) rows from {nseq} of {w.B} sequences, scaled to all "
              + f"rows; masks and acceptance on all {w.B} sequences; fp64 oracle, OpenMP")
    return per_step, sample, cores


def run_reference(args, w, idx):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = make_inputs(w, 1000 + idx, with_kv=False)
    per_step, sample, cores = time_oracle(inp, budget_s=90.0, steps=args.steps,
                                          warmup=args.warmup)
    value = w.B * w.N / per_step
    line = {
        "impl": "reference", "metric": "verified tree-nodes/s per attn layer", "value": value,
        "unit": "nodes/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, page_size=None):
    c = {"workload": w.name, "B": w.B, "N": w.N,
         "context": w.L if w.L_hi is None else f"U[{w.L},{w.L_hi}]", "Hq": w.Hq,
         "Hkv": w.Hkv, "head_dim": w.D, "vocab": w.V, "tree": w.tree}
    if page_size is not None:
        c["page_size"] = page_size
    return c


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class StepRunner:
    """Device inputs (rotated over enough copies to exceed L2), outputs and the
    three calls of one verify step for one workload."""

    def __init__(self, sv, torch, w, inp, dev):
        self.sv, self.torch, self.w, self.inp, self.dev = sv, torch, w, inp, dev
        bf = w.dtype == "bf16"

        def to_dev(x, as_bf16=False):
            t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if as_bf16 else x).to(dev)
            return t.view(torch.bfloat16) if as_bf16 else t

        self.base = {
            "q": to_dev(inp.q, bf), "k": to_dev(inp.k_cache, bf), "v": to_dev(inp.v_cache, bf),
            "page_table": to_dev(inp.page_table), "seq_lens": to_dev(inp.seq_lens),
            "parent": to_dev(inp.parent), "tokens": to_dev(inp.tokens),
            "target": to_dev(inp.target), "draft": to_dev(inp.draft),
            "u_accept": to_dev(inp.u_accept), "u_bonus": to_dev(inp.u_bonus),
        }
        self.step_bytes = sum(t.numel() * t.element_size() for t in self.base.values())
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.nsets = max(1, math.ceil(3 * self.l2 / self.step_bytes))
        self.sets = [self.base] + [{k: v.clone() for k, v in self.base.items()}
                                   for _ in range(self.nsets - 1)]
        B, N, Hq, D = w.B, w.N, w.Hq, w.D
        self.anc = torch.empty((B, N, 1), dtype=torch.int64, device=dev)
        self.depth = torch.empty((B, N), dtype=torch.int32, device=dev)
        self.mstat = torch.empty((B,), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.base["q"])
        self.lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
        self.astat = torch.empty((B,), dtype=torch.int32, device=dev)
        self.attn_ws_need = sv.tree_verify_attn_workspace_size(
            B, N, Hq, w.Hkv, D, self.base["q"].dtype, inp.page_table.shape[1], inp.page_size)
        # zero-filled once; every call leaves it so
        self.attn_ws = torch.zeros((max(self.attn_ws_need, 1),), dtype=torch.uint8, device=dev)
        self.acc_ws_need = sv.spec_accept_workspace_size(B, N, w.V)
        self.acc_ws = torch.empty((self.acc_ws_need,), dtype=torch.uint8, device=dev)
        self.acc_out = {}
        self.cap = torch.cuda.Stream(dev)

    def mask_call(self, s):
        self.sv.tree_mask_build(s["parent"], self.anc, self.depth, self.mstat)

    def attn_call(self, s):
        # ancestor masks and attention in one call (one kernel for bf16)
        self.sv.tree_mask_attn(s["parent"], s["q"], s["k"], s["v"], s["page_table"],
                               s["seq_lens"], anc=self.anc, depth=self.depth,
                               mask_status=self.mstat, out=self.out, lse=self.lse,
                               workspace=self.attn_ws, status=self.astat)

    def accept_call(self, s):
        self.sv.spec_accept(s["target"], s["draft"], s["tokens"], s["parent"], s["u_accept"],
                            s["u_bonus"], workspace=self.acc_ws, outputs=self.acc_out)

    def step(self, s):
        self.attn_call(s)
        self.accept_call(s)

    def launches_per_step(self):
        # fused masks + attention: one kernel for bf16, mask + attention for fp32
        attn = 1 if self.w.dtype == "bf16" else 2
        return attn + (2 if self.acc_ws_need > 0 else 1)

    def capture(self, fn, s):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.cap):
            fn(s)
        return g

    def capture_instrumented(self, s):
        """The step graph with a timing event before, between and after its two
        calls (events of external kind, so that replays can be timed), or None
        where this PyTorch cannot record such events in a graph."""
        torch = self.torch
        try:
            evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
        except TypeError:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.cap):
            evs[0].record()
            self.attn_call(s)
            evs[1].record()
            self.accept_call(s)
            evs[2].record()
        return g, evs

    def check(self):
        self.torch.cuda.synchronize(self.dev)
        assert int(self.astat.abs().sum()) == 0 and int(self.acc_out["status"].abs().sum()) == 0
        assert int(self.mstat.abs().sum()) == 0
        assert bool(self.torch.isfinite(self.out.float()).all())

    def free(self):
        self.sets = self.base = None
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def time_step(r: StepRunner, steps, warmup, barrier, stream, clk=None):
    """Step time from replays of one CUDA graph per input set, and per-kernel
    times inside the step from the instrumented capture.

    Returns a dict: ``ms`` per step (plain graphs), ``in_step`` ms of the
    fused masks + attention call (with its split merge) and of the acceptance
    call, and their total inside one instrumented step (its events sit
    between the kernels, so the dependent-launch overlap of the plain graph
    is lost there), and ``single_call`` ms of each call captured and
    replayed alone (the stand-alone mask build included)."""
    torch = r.torch
    for i in range(warmup):
        r.step(r.sets[i % r.nsets])
    barrier()
    g_step = [r.capture(r.step, s) for s in r.sets]
    barrier()
    for i in range(warmup):
        g_step[i % r.nsets].replay()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        # keep the GPU busy until the sampler reports (nvidia-smi starts in ~0.1-0.5 s)
        t_soak = time.perf_counter()
        i = 0
        n0 = len(clk.lines)
        while (len(clk.lines) < n0 + 3 and time.perf_counter() - t_soak < 5.0) or i < warmup:
            g_step[i % r.nsets].replay()
            i += 1
            if i % 16 == 0:
                torch.cuda.synchronize(r.dev)
        barrier()
    t_start.record(stream)
    for i in range(steps):
        g_step[i % r.nsets].replay()
    t_end.record(stream)
    barrier()
    ms = t_start.elapsed_time(t_end) / steps
    res = {"ms": ms}
    # per-kernel times inside the step
    inst = [r.capture_instrumented(s) for s in r.sets]
    if inst[0] is not None:
        acc = np.zeros(3)
        for i in range(steps):
            g, evs = inst[i % r.nsets]
            g.replay()
            torch.cuda.synchronize(r.dev)
            acc += [evs[0].elapsed_time(evs[1]), evs[1].elapsed_time(evs[2]),
                    evs[0].elapsed_time(evs[2])]
        acc /= steps
        res["in_step"] = {"attn_ms": acc[0], "accept_ms": acc[1], "total_ms": acc[2],
                          "method": "timing events captured between the calls of the step "
                                    "graph; replayed per input set"}
    # each call captured alone, replayed back to back with events around it
    single = {}
    for name, fn in (("mask", r.mask_call), ("attn", r.attn_call), ("accept", r.accept_call)):
        gs = [r.capture(fn, s) for s in r.sets]
        barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            evs[i][0].record(stream)
            gs[i % r.nsets].replay()
            evs[i][1].record(stream)
        barrier()
        single[name + "_ms"] = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    res["single_call"] = single
    if "in_step" not in res:
        res["in_step"] = {"attn_ms": single["attn_ms"], "accept_ms": single["accept_ms"],
                          "total_ms": single["attn_ms"] + single["accept_ms"],
                          "method": "single-call graphs (this PyTorch records no timing "
                                    "events inside a graph)"}
    g_step.clear()
    return res


def time_lm_head(sv, torch, w, dev, steps, peak, fused_inputs=None):
    """The LM head of the workload's target layer: R = B*N hidden rows of size
    H = Hq*D (the model's hidden size) against a [V, H] bf16 weight, fp32
    logits out; each call timed alone with CUDA events, the L2 flushed
    between calls. With ``fused_inputs`` (draft logits, tokens, parent,
    uniforms on the device) the fused LM head + walk call is timed too."""
    R, H, V = w.B * w.N, w.Hq * w.D, w.V
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321)
    hidden = torch.randn((w.B, w.N, H), generator=gen, device=dev).to(torch.bfloat16)
    weight = (torch.randn((V, H), generator=gen, device=dev) * (3.0 / math.sqrt(H))).to(
        torch.bfloat16)
    logits = torch.empty((w.B, w.N, V), dtype=torch.float32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in ts) / steps

    ms = timed(lambda: sv.lm_head(hidden, weight, logits=logits, status=status))
    assert int(status.item()) == 0 and bool(torch.isfinite(logits).all())
    burst, sustained, kind = measured_tensor_peak()
    flops = 2.0 * R * H * V
    nbytes = V * H * 2 + R * H * 2 + R * V * 4
    out = {"ms": ms, "R": R, "H": H, "V": V, "flops": flops, "tflops": flops / ms / 1e9,
           "frac_of_bf16_sustained": flops / ms / 1e9 / sustained,
           "frac_of_bf16_burst": flops / ms / 1e9 / burst, "peak_kind": kind,
           "bytes": nbytes, "gbs": nbytes / ms / 1e6, "frac_of_hbm": nbytes / ms / 1e6 / peak,
           "bytes_note": "weight read once, hidden states read, fp32 logits written",
           "inputs": "seeded random bf16 hidden states N(0,1) and weight N(0, 9/H)"}
    if fused_inputs is not None:
        fo = {}
        f = fused_inputs
        ms_f = timed(lambda: sv.spec_accept_lmhead(hidden, weight, f["draft"], f["tokens"],
                                                   f["parent"], f["u_accept"], f["u_bonus"],
                                                   outputs=fo))
        assert int(fo["status"].abs().sum()) == 0 and int(fo["lm_status"].item()) == 0
        out["fused_with_walk_ms"] = ms_f
    del hidden, weight, logits, flush
    torch.cuda.empty_cache()
    return out


def time_graph_of_steps(r: StepRunner, stream, barrier, n=100) -> float:
    """Launch-amortised ms per step: ``n`` consecutive steps (rotating input
    sets) captured as one CUDA graph, replayed after one warm-up replay."""
    torch = r.torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=r.cap):
        for i in range(n):
            r.step(r.sets[i % r.nsets])
    g.replay()
    barrier()
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    g.replay()
    h1.record(stream)
    barrier()
    ms = h0.elapsed_time(h1) / n
    # a second replay for short steps, whose single replay is only a few ms
    if ms < 1.0:
        h0.record(stream)
        for _ in range(3):
            g.replay()
        h1.record(stream)
        barrier()
        ms = h0.elapsed_time(h1) / (3 * n)
    del g
    return ms


def workload_summary(r: StepRunner, t: dict, peak, clocks):
    """Attention and acceptance times of one workload with their roofline shares."""
    w, inp = r.w, r.inp
    nb = algorithmic_bytes(w, inp.seq_lens, inp.parent)
    path = r.acc_out["path"].cpu().numpy()
    alen = r.acc_out["accept_len"].cpu().numpy()
    acc_bytes = walk_bytes(w, inp.parent, path, alen)
    nodes = visited_nodes(alen)
    ins = t["in_step"]
    attn_gbs = nb["attn_bytes"] / (ins["attn_ms"] / 1e3) / 1e9
    acc_gbs = acc_bytes / (ins["accept_ms"] / 1e3) / 1e9
    return {
        "config": workload_config(w, inp.page_size),
        "step_us": t["ms"] * 1e3,
        "nodes_per_s": w.B * w.N / (t["ms"] / 1e3),
        "attn_us": ins["attn_ms"] * 1e3,
        "attn_bytes": nb["attn_bytes"],
        "attn_frac_of_hbm": attn_gbs / peak,
        "accept_us": ins["accept_ms"] * 1e3,
        "accept_bytes": acc_bytes,
        "accept_frac_of_hbm": acc_gbs / peak,
        "accept_bytes_all_rows": nb["accept_bytes"],
        "accept_visited_nodes": nodes,
        "accept_us_per_visited_node": ins["accept_ms"] * 1e3 / nodes,
        "accept_us_per_visited_node_per_sequence": ins["accept_ms"] * 1e3 * w.B / nodes,
        "mask_alone_us": t["single_call"]["mask_ms"] * 1e3,
        "in_step_total_us": ins["total_ms"] * 1e3,
        "single_call_us": {k.replace("_ms", ""): v * 1e3 for k, v in t["single_call"].items()},
        "clocks": clocks,
    }


def run_ours(args, w, idx):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from speculative_decoding_tree_03_gb300 import build as _build
    _build.build()
    import speculative_decoding_tree_03_gb300 as sv
    if args.attn_chunks:
        assert sv.load_library().svf_debug_set_attn_splits(args.attn_chunks) == 0
    if args.attn_kernel:
        assert sv.load_library().svf_debug_set_attn_kernel(args.attn_kernel) == 0

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- the other workloads first (small, freed afterwards), rank 0 only
    per_workload = {}
    if not args.no_per_workload and rank == 0:
        for j, w2 in enumerate(WORKLOADS):
            if w2.name == w.name:
                continue
            inp2 = make_inputs(w2, 1000 + j)
            r2 = StepRunner(sv, torch, w2, inp2, dev)
            with ClockSampler(local) as clk2:
                t2 = time_step(r2, args.steps, args.warmup, lambda: torch.cuda.synchronize(dev),
                               stream, clk2)
                # a few more samples under load
                t_tail = time.perf_counter()
                n0 = len(clk2.lines)
                while len(clk2.lines) < n0 + 2 and time.perf_counter() - t_tail < 2.0:
                    for _ in range(16):
                        r2.step(r2.sets[0])
                    torch.cuda.synchronize(dev)
            r2.check()
            per_workload[w2.name] = workload_summary(r2, t2, peak, clk2.summary())
            g100_ms = time_graph_of_steps(r2, stream, lambda: torch.cuda.synchronize(dev))
            per_workload[w2.name]["graph_100_steps"] = {
                "step_us": g100_ms * 1e3, "nodes_per_s": w2.B * w2.N / (g100_ms / 1e3),
                "note": "100 steps captured as one CUDA graph"}
            if w2.dtype == "bf16":
                per_workload[w2.name]["lm_head"] = time_lm_head(sv, torch, w2, dev,
                                                                args.steps, peak)
            r2.free()
            del r2, inp2

    seed = 1000 + idx
    inp = make_inputs(w, seed)
    nb = algorithmic_bytes(w, inp.seq_lens, inp.parent)
    r = StepRunner(sv, torch, w, inp, dev)
    B, N, Hq, D = w.B, w.N, w.Hq, w.D
    bf = w.dtype == "bf16"

    with ClockSampler(local) as clk:
        t = time_step(r, args.steps, args.warmup, barrier, stream, clk)
        t_tail = time.perf_counter()
        n0 = len(clk.lines)
        while len(clk.lines) < n0 + 2 and time.perf_counter() - t_tail < 2.0:
            r.step(r.sets[0])
            torch.cuda.synchronize(dev)
    r.check()
    ms_local = t["ms"]
    ins = t["in_step"]

    # launch-amortised: 100 consecutive steps captured as one CUDA graph
    ms100_local = time_graph_of_steps(r, stream, barrier)

    def timed_calls(fn, name_out=None):
        """ms per call of ``fn`` captured alone per input set, replayed K times."""
        fn(r.sets[0])
        barrier()
        graphs = [r.capture(fn, s) for s in r.sets]
        barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            evs[i][0].record(stream)
            graphs[i % r.nsets].replay()
            evs[i][1].record(stream)
        barrier()
        return sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps

    # ---- KV commit of the accepted path (one layer), timed on its own after
    # the step: it rewrites tree rows of the cache in place, which later
    # replays of the step read as ordinary (finite) K/V
    commit_out = {}
    acc_out = r.acc_out

    def commit_call(s):
        sv.kv_commit(s["k"], s["v"], s["page_table"], s["seq_lens"], acc_out["path"],
                     acc_out["accept_len"], outputs=commit_out)

    commit_ms = timed_calls(commit_call)
    assert int(commit_out["status"].abs().sum()) == 0

    # ---- the target-only acceptance variants on the same inputs, each timed
    # on its own (greedy argmax matching; one-hot candidate sampling)
    var_out = {"greedy": {}, "onehot": {}, "bf16": {}, "greedy_bf16": {}, "onehot_bf16": {}}

    def greedy_call(s):
        sv.spec_accept_greedy(s["target"], s["tokens"], s["parent"], outputs=var_out["greedy"])

    def onehot_call(s):
        sv.spec_accept_onehot(s["target"], s["tokens"], s["parent"], s["u_accept"],
                              s["u_bonus"], outputs=var_out["onehot"])

    # ---- EAGLE-2 tree construction for this workload's batch and vocabulary:
    # k = 8 per round, 6 rounds, N nodes kept, from seeded synthetic draft rows
    e2k, e2rounds = 8, 6
    e2gen = torch.Generator(device=dev)
    e2gen.manual_seed(1234)
    e2rows = [torch.randn((B, 1 if rr == 0 else e2k, w.V), generator=e2gen, device=dev) * 2.0
              for rr in range(e2rounds)]
    e2roots = torch.zeros((B,), dtype=torch.int32, device=dev)
    e2cap = 1 + e2k + (e2rounds - 1) * e2k * e2k
    e2pool = sv.eagle2_pool(e2roots, e2cap)
    e2f0 = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    e2fr = [torch.empty((B, e2k), dtype=torch.int32, device=dev) for _ in range(e2rounds)]
    e2out = {}

    def eagle2_call(s):
        sv.eagle2_init(e2pool, e2roots)
        f = e2f0
        for rr in range(e2rounds):
            f = sv.eagle2_expand(e2pool, e2rows[rr], f, e2k, next_frontier=e2fr[rr])
        return sv.eagle2_finalize(e2pool, N, outputs=e2out)

    # the walk on bf16 copies of the logits (one input set: larger than L2)
    bf_logits = {k: r.sets[0][k].to(torch.bfloat16) for k in ("target", "draft")}

    def bf16_call(s):
        sv.spec_accept(bf_logits["target"], bf_logits["draft"], s["tokens"], s["parent"],
                       s["u_accept"], s["u_bonus"], outputs=var_out["bf16"])

    def greedy_bf16_call(s):
        sv.spec_accept_greedy(bf_logits["target"], s["tokens"], s["parent"],
                              outputs=var_out["greedy_bf16"])

    def onehot_bf16_call(s):
        sv.spec_accept_onehot(bf_logits["target"], s["tokens"], s["parent"], s["u_accept"],
                              s["u_bonus"], outputs=var_out["onehot_bf16"])

    lm = time_lm_head(sv, torch, w, dev, args.steps, peak, fused_inputs=r.base) \
        if bf else None

    var_ms = {}
    for name, fn in (("greedy", greedy_call), ("onehot", onehot_call), ("eagle2", eagle2_call),
                     ("bf16", bf16_call), ("greedy_bf16", greedy_bf16_call),
                     ("onehot_bf16", onehot_bf16_call)):
        var_ms[name] = timed_calls(fn)
        if name != "eagle2":
            assert int(var_out[name]["status"].abs().sum()) == 0
    assert int(e2out["n_out"].min()) == min(N, e2cap)
    del e2rows, bf_logits

    def rmax(x):
        if world == 1:
            return x
        tt = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())

    def rsum(x):
        if world == 1:
            return x
        tt = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.SUM)
        return float(tt.item())

    ms, value = aggregate(ms_local, B * N, world, rmax, rsum)
    ms100 = rmax(ms100_local)

    # ---- end to end through the public API from pinned host buffers. The
    # KV cache of the prefix is device-resident state (written once, as a
    # serving loop keeps it); a step's inputs are everything else: the
    # queries, the K/V rows of the tree's own tokens (scattered into their
    # cache slots on arrival), the tree, the uniforms, the lengths and page
    # table, and both logits arrays. They sit in one pinned host buffer and
    # travel in one copy into one of two device buffers whose slices the
    # step's tensors view; a side stream copies step i + 1 while step i runs
    # (double buffering), and every step's outputs come back to pinned host
    # memory.
    base = r.base
    # the outputs of one device-resident step on these inputs: the end-to-end
    # steps must reproduce them bit for bit
    r.step(base)
    torch.cuda.synchronize(dev)
    ref_out = r.out.clone().cpu()
    ref_res = {k: acc_out[k].clone().cpu() for k in ("accept_len", "path", "out_tokens", "status")}
    kres, vres = base["k"], base["v"]
    Hkv, D = kres.shape[2], kres.shape[3]
    ps = int(inp.page_size)
    slots = np.empty((B * N,), np.int64)
    for b in range(B):
        pos = int(inp.seq_lens[b]) + np.arange(N)
        slots[b * N:(b + 1) * N] = inp.page_table[b, pos // ps].astype(np.int64) * ps + pos % ps
    kflat_h = kres.view(-1, Hkv, D)
    slots_d = torch.from_numpy(slots).to(dev)
    step_in = {k: v for k, v in base.items() if k not in ("k", "v")}
    step_in["tree_k"] = kflat_h.index_select(0, slots_d)
    step_in["tree_v"] = vres.view(-1, Hkv, D).index_select(0, slots_d)
    step_in["slots"] = slots_d
    offs, total = {}, 0
    for k, v in step_in.items():
        nbytes = v.numel() * v.element_size()
        offs[k] = (total, nbytes, v.shape, v.dtype)
        total += (nbytes + 255) & ~255
    host_in = torch.empty((total,), dtype=torch.uint8).pin_memory()
    for k, (o, nbytes, _, _) in offs.items():
        host_in[o:o + nbytes].copy_(step_in[k].reshape(-1).view(torch.uint8).cpu())
    del step_in
    # the rotated input copies are no longer needed: make room for the two
    # end-to-end device buffers (the resident cache stays)
    r.sets = [r.base]
    torch.cuda.empty_cache()
    dbufs = [torch.empty((total,), dtype=torch.uint8, device=dev) for _ in range(2)]
    dsets = [{k: buf[o:o + nbytes].view(dt).view(shape)
              for k, (o, nbytes, shape, dt) in offs.items()} for buf in dbufs]
    for ds in dsets:
        ds["k"], ds["v"] = kres, vres
    h2d = sum(nbytes for _, nbytes, _, _ in offs.values())
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    res_h = {k: torch.empty((B, N) if k in ("path", "out_tokens") else (B,),
                            dtype=torch.int32).pin_memory()
             for k in ("accept_len", "path", "out_tokens", "status")}
    d2h = out_h.numel() * out_h.element_size() + sum(tt.numel() * 4 for tt in res_h.values())
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in dbufs]
    used = [torch.cuda.Event() for _ in dbufs]

    def issue_copy(i):
        j = i % len(dbufs)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(used[j])  # the step that last read buffer j
            dbufs[j].copy_(host_in, non_blocking=True)
            copied[j].record(copy_stream)

    def e2e_run(steps, e_start=None):
        if e_start is not None:
            copy_stream.wait_event(e_start)
        issue_copy(0)
        for i in range(steps):
            if i + 1 < steps:
                issue_copy(i + 1)
            j = i % len(dbufs)
            stream.wait_event(copied[j])
            ds = dsets[j]
            # the tree's K/V rows into their cache slots, then the step
            kres.view(-1, Hkv, D).index_copy_(0, ds["slots"], ds["tree_k"])
            vres.view(-1, Hkv, D).index_copy_(0, ds["slots"], ds["tree_v"])
            r.step(ds)
            used[j].record(stream)
            out_h.copy_(r.out, non_blocking=True)
            for k in res_h:
                res_h[k].copy_(acc_out[k], non_blocking=True)

    e2e_run(min(args.warmup, 3))
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, e0)
    e1.record(stream)
    barrier()
    e2e_ms = rmax(e0.elapsed_time(e1) / args.steps)
    e2e_value = rsum(B * N) / (e2e_ms / 1e3)
    r.check()
    torch.cuda.synchronize(dev)
    assert torch.equal(out_h.view(torch.int16) if out_h.dtype == torch.bfloat16 else out_h,
                       ref_out.view(torch.int16) if ref_out.dtype == torch.bfloat16 else ref_out), \
        "end-to-end attention output differs from the device-resident step"
    for k, v in ref_res.items():
        assert torch.equal(res_h[k], v), f"end-to-end {k} differs from the device-resident step"

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    head = workload_summary(r, t, peak, clk.summary())
    attn_ms = ins["attn_ms"]
    acc_ms = ins["accept_ms"]
    attn_gbs = nb["attn_bytes"] / (attn_ms / 1e3) / 1e9
    acc_bytes = head["accept_bytes"]
    acc_gbs = acc_bytes / (acc_ms / 1e3) / 1e9
    path_h = acc_out["path"].cpu().numpy()
    alen_h = acc_out["accept_len"].cpu().numpy()
    rows_moved = int(sum(int((path_h[b, 1: alen_h[b] + 1] != np.arange(1, alen_h[b] + 1)).sum())
                         for b in range(B)))
    commit_bytes = rows_moved * w.Hkv * D * (2 if bf else 4) * 2 * 2
    commit_gbs = commit_bytes / (commit_ms / 1e3) / 1e9
    e2bytes = (1 + (e2rounds - 1) * e2k) * B * w.V * 4
    var_kernels = {"eagle2_build": {
        "ms": var_ms["eagle2"], "bytes": e2bytes, "gbs": e2bytes / (var_ms["eagle2"] / 1e3) / 1e9,
        "frac_of_hbm": e2bytes / (var_ms["eagle2"] / 1e3) / 1e9 / peak,
        "config": f"k={e2k}, {e2rounds} rounds, N={N}, B={B}, V={w.V}: init, {e2rounds} "
                  f"expansions, rerank",
        "bytes_note": "draft rows read by the expansions"}}
    bp = var_out["bf16"]["path"].cpu().numpy()
    bl = var_out["bf16"]["accept_len"].cpu().numpy()
    bfb = walk_bytes(w, inp.parent, bp, bl) // 2
    var_kernels["spec_accept_bf16"] = {
        "ms": var_ms["bf16"], "bytes": bfb, "gbs": bfb / (var_ms["bf16"] / 1e3) / 1e9,
        "frac_of_hbm": bfb / (var_ms["bf16"] / 1e3) / 1e9 / peak,
        "bytes_note": "bf16 rows of the visited nodes (the logits rounded to bf16)"}
    for name in ("greedy", "onehot", "greedy_bf16", "onehot_bf16"):
        vp = var_out[name]["path"].cpu().numpy()
        vl = var_out[name]["accept_len"].cpu().numpy()
        vb = sum(int(vl[b]) + 1 for b in range(B)) * w.V * (2 if name.endswith("bf16") else 4)
        var_kernels["spec_accept_" + name] = {
            "ms": var_ms[name], "bytes": vb, "gbs": vb / (var_ms[name] / 1e3) / 1e9,
            "frac_of_hbm": vb / (var_ms[name] / 1e3) / 1e9 / peak,
            "mean_accept_len": float(vl.mean()),
            "bytes_note": "target rows of the visited nodes"}
        assert (vp[:, 0] == 0).all()
    line = {
        "metric": "verified tree-nodes/s per attn layer",
        "value": value,
        "unit": "nodes/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if bf else "f32",
        "data": "synthetic",
        "config": {
            **workload_config(w, inp.page_size),
            "l2": f"inputs rotate over {r.nsets} copies ({r.nsets * r.step_bytes / 1e6:.0f} MB "
                  f"> L2 {r.l2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": "one CUDA graph per step: masks + attention (one fused call), acceptance",
            "attn_chunks": args.attn_chunks or "library's choice",
            "attn_kernel": {0: "library's choice", 1: "chunks merged in clusters",
                            2: "persistent, one CTA per SM"}[args.attn_kernel],
            "e2e_copies": "the prefix KV cache resident on the device; per step one packed "
                          "pinned host-to-device copy of the step's inputs (queries, the tree's "
                          "K/V rows, tree, uniforms, lengths, page table, both logits arrays), "
                          "issued one step ahead on a side stream; outputs read back every step",
        },
        "accept_steps_per_s": rsum(B) / (ms / 1e3),
        "graph_100_steps": {"ms_per_step": ms100, "value": rsum(B * N) / (ms100 / 1e3),
                            "note": "100 steps captured as one CUDA graph"},
        "in_step": {"attn_us": attn_ms * 1e3,
                    "accept_us": acc_ms * 1e3, "total_us": ins["total_ms"] * 1e3,
                    "step_us": ms * 1e3, "method": ins["method"],
                    "note": "the plain step graph launches its kernels with programmatic "
                            "dependent launch; events between them serialise the calls, so "
                            "total_us is at least step_us"},
        "kernels": {
            "tree_verify_attn": {"ms": attn_ms, "bytes": nb["attn_bytes"], "gbs": attn_gbs,
                                 "frac_of_hbm": attn_gbs / peak,
                                 "single_call_ms": t["single_call"]["attn_ms"]},
            "spec_accept": {"ms": acc_ms, "bytes": acc_bytes, "gbs": acc_gbs,
                            "frac_of_hbm": acc_gbs / peak,
                            "single_call_ms": t["single_call"]["accept_ms"],
                            "visited_nodes": head["accept_visited_nodes"],
                            "us_per_visited_node": head["accept_us_per_visited_node"],
                            "us_per_visited_node_per_sequence":
                                head["accept_us_per_visited_node_per_sequence"],
                            "bytes_all_rows": nb["accept_bytes"],
                            "bytes_note": "rows of the visited nodes; bytes_all_rows counts "
                                          "every row a walk could test"},
            "tree_mask_build": {"in_step": "built inside the fused attention call",
                                "single_call_ms": t["single_call"]["mask_ms"],
                                "note": "svf_tree_mask_build alone, captured and replayed"},
            "kv_commit": {"ms": commit_ms, "bytes": commit_bytes, "gbs": commit_gbs,
                          "frac_of_hbm": commit_gbs / peak, "rows_moved": rows_moved,
                          "bytes_note": "K and V rows of accepted nodes not yet in place, "
                                        "read and written, one layer"},
            **var_kernels,
            **({"lm_head": lm} if lm is not None else {}),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "tree_verify_attn",
            "achieved": attn_gbs,
            "peak": peak,
            "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
            "unit": "GB/s",
            "frac": attn_gbs / peak,
            "traffic": (committed_traffic(w.name, args.attn_chunks)
                        if not args.batch and not args.attn_kernel else None),
            "duration_from": "CUDA events around the attention call inside the step graph",
        },
        "per_workload": per_workload,
        "e2e": {"value": e2e_value, "unit": "nodes/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": r.launches_per_step() * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        per_step, sample, cores = time_oracle(inp)
        line["cpu_baseline"] = {"value": B * N / per_step, "unit": "nodes/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--attn-kernel", type=int, default=0, choices=[0, 1, 2],
                    help="bf16 attention kernel: 0 the library's choice, 1 KV chunks merged in "
                         "thread-block clusters, 2 persistent (one CTA per SM)")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this many sequences instead of its own batch "
                         "(a smaller case of the same shapes, for profiler captures)")
    ap.add_argument("--attn-chunks", type=int, default=0,
                    help="KV chunks per (sequence, KV head) of the bf16 attention, 1..8 "
                         "(0: the library's choice); 1 launches no thread-block cluster")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    idx, w = workload_by_name(args.workload)
    if args.batch > 0:
        w = dataclasses.replace(w, B=args.batch)
    if args.impl == "reference":
        run_reference(args, w, idx)
    else:
        run_ours(args, w, idx)


if __name__ == "__main__":
    main()
