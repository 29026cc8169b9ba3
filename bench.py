"""Benchmark of one verify step: ancestor masks -> tree attention (one layer) ->
acceptance walk, on synthetic inputs shaped like the workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

Prints ONE JSON line on rank 0. ``value`` is verified tree nodes per second
(per attention layer) over all ranks, with inputs resident in HBM; ``e2e``
repeats the measurement through the public API from pinned host buffers with
the copies inside the timed region (one packed host-to-device copy per step,
issued on a side stream one step ahead, and the outputs read back). Between timed steps the inputs rotate over
enough copies that the working set exceeds L2. ``--impl reference`` times the
fp64 CPU oracle on the host cores instead (the reference arm).

Multi-GPU: the path does not shard; each rank runs an independent replica of
the workload (weak scaling) and the step time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
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

DEFAULT_WORKLOAD = "binary_tree_8b"
FALLBACK_HBM_GBS = 6800.0


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


def source_hash(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(workload, kernel_src):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    has not changed since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("source_hash") == source_hash(kernel_src):
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

def _oracle_inputs(inp):
    """Logical float32 K/V, q for the oracle (regenerated from the generator)."""
    from synth.gen import logical_kv, bf16_bits_to_f32
    w = inp.w
    T = inp.seq_lens.astype(np.int64) + w.N
    Tcap = int(T.max())
    K = np.zeros((w.B, Tcap, w.Hkv, w.D), np.float32)
    V = np.zeros_like(K)
    cvt = (lambda x: bf16_bits_to_f32(x)) if w.dtype == "bf16" else (lambda x: x)
    for b in range(w.B):
        for g in range(w.Hkv):
            k, v = logical_kv(w, inp.seed, b, g, int(T[b]))
            K[b, : T[b], g] = cvt(k)
            V[b, : T[b], g] = cvt(v)
    return cvt(inp.q), K, V


def time_oracle(inp, budget_s=15.0, max_steps=20, steps=None, warmup=0, threads=None):
    """Time the fp64 oracle for the whole verify step on the host cores.

    Without ``steps``: as many steps as fit in ``budget_s`` (at most
    ``max_steps``). With ``steps``: ``warmup`` untimed steps, then exactly
    ``steps`` timed ones, the attention rows sampled so that all of them fit
    in ``budget_s``. Returns (seconds per step, sample text, cores)."""
    import oracle
    w = inp.w
    cores = threads or len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    q, K, V = _oracle_inputs(inp)
    rows_all = w.B * w.N * w.Hq
    # time one row first to size the sample
    t0 = time.perf_counter()
    oracle.tree_attn(q, K, V, inp.seq_lens, inp.parent, rows=np.array([[0, 0, 0]]))
    one = max(time.perf_counter() - t0, 1e-6)
    frac = 1.0
    rows = None
    per_step_budget = budget_s / 2 if steps is None else budget_s / max(1, steps + warmup)
    if one * rows_all / cores > per_step_budget:
        nsel = max(cores, int(per_step_budget * cores / one))
        sel = np.linspace(0, rows_all - 1, nsel).astype(np.int64)
        rows = np.stack([sel // (w.N * w.Hq), (sel // w.Hq) % w.N, sel % w.Hq], 1)
        frac = nsel / rows_all
    def one_step():
        oracle.tree_attn(q, K, V, inp.seq_lens, inp.parent, rows=rows)
        oracle.tree_mask(inp.parent)
        oracle.spec_accept(inp.target, inp.draft, inp.tokens, inp.parent, inp.u_accept,
                           inp.u_bonus)

    for _ in range(warmup):
        one_step()
    fixed = steps
    steps = 0
    t_attn = t_acc = 0.0
    start = time.perf_counter()
    while ((fixed is not None and steps < fixed) or
           (fixed is None and steps < max_steps and
            (steps == 0 or time.perf_counter() - start < budget_s))):
        t0 = time.perf_counter()
        oracle.tree_attn(q, K, V, inp.seq_lens, inp.parent, rows=rows)
        t1 = time.perf_counter()
        oracle.tree_mask(inp.parent)
        oracle.spec_accept(inp.target, inp.draft, inp.tokens, inp.parent, inp.u_accept,
                           inp.u_bonus)
        t2 = time.perf_counter()
        t_attn += (t1 - t0) / frac
        t_acc += t2 - t1
        steps += 1
    per_step = (t_attn + t_acc) / steps
    sample = ((f"{warmup} untimed + " if warmup else "")
              + f"{steps} timed verify step(s) of {w.name}; attention "
              + ("all rows" if rows is None else f"{len(rows)} of {rows_all} rows, scaled")
              + "; fp64 oracle, OpenMP")
    return per_step, sample, cores


def run_reference(args, w, idx):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = make_inputs(w, 1000 + idx)
    per_step, sample, cores = time_oracle(inp, budget_s=90.0, steps=args.steps,
                                          warmup=args.warmup)
    value = w.B * w.N / per_step
    line = {
        "impl": "reference", "metric": "verified tree-nodes/s per attn layer", "value": value,
        "unit": "nodes/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "context": w.L, "Hq": w.Hq,
                   "Hkv": w.Hkv, "head_dim": w.D, "vocab": w.V},
        "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

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

    seed = 1000 + idx
    inp = make_inputs(w, seed)
    nb = algorithmic_bytes(w, inp.seq_lens, inp.parent)
    dev = torch.device("cuda", local)

    def to_dev(x, bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if bf16 else x).to(dev)
        return t.view(torch.bfloat16) if bf16 else t

    bf = w.dtype == "bf16"
    base = {
        "q": to_dev(inp.q, bf), "k": to_dev(inp.k_cache, bf), "v": to_dev(inp.v_cache, bf),
        "page_table": to_dev(inp.page_table), "seq_lens": to_dev(inp.seq_lens),
        "parent": to_dev(inp.parent), "tokens": to_dev(inp.tokens),
        "target": to_dev(inp.target), "draft": to_dev(inp.draft),
        "u_accept": to_dev(inp.u_accept), "u_bonus": to_dev(inp.u_bonus),
    }
    step_bytes = sum(t.numel() * t.element_size() for t in base.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(1, math.ceil(3 * l2 / step_bytes))
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]

    B, N, Hq, D = w.B, w.N, w.Hq, w.D
    stream = torch.cuda.current_stream(dev)
    anc = torch.empty((B, N, 1), dtype=torch.int64, device=dev)
    depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    mstat = torch.empty((B,), dtype=torch.int32, device=dev)
    out = torch.empty_like(base["q"])
    lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    astat = torch.empty((B,), dtype=torch.int32, device=dev)
    ws_need = sv.tree_verify_attn_workspace_size(B, N, Hq, w.Hkv, D, base["q"].dtype,
                                                 inp.page_table.shape[1], inp.page_size)
    attn_ws = torch.empty((max(ws_need, 1),), dtype=torch.uint8, device=dev)
    acc_ws = torch.empty((sv.spec_accept_workspace_size(B, N, w.V),), dtype=torch.uint8,
                         device=dev)
    acc_out = {}

    def mask_call(s):
        sv.tree_mask_build(s["parent"], anc, depth, mstat)

    def attn_call(s):
        sv.tree_verify_attn(s["q"], s["k"], s["v"], s["page_table"], s["seq_lens"], anc,
                            out=out, lse=lse, workspace=attn_ws, status=astat)

    def accept_call(s):
        sv.spec_accept(s["target"], s["draft"], s["tokens"], s["parent"], s["u_accept"],
                       s["u_bonus"], workspace=acc_ws, outputs=acc_out)

    def step(s):
        mask_call(s)
        attn_call(s)
        accept_call(s)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        step(sets[i % nsets])
    barrier()
    # Each step is issued as one CUDA graph (as a serving loop replays its
    # decode step); per-kernel times come from graphs of the single calls.
    cap = torch.cuda.Stream(dev)

    def capture(fn, s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn(s)
        return g

    g_step = [capture(step, s) for s in sets]
    g_mask = [capture(mask_call, s) for s in sets]
    g_attn = [capture(attn_call, s) for s in sets]
    g_acc = [capture(accept_call, s) for s in sets]
    barrier()
    for i in range(args.warmup):
        g_step[i % nsets].replay()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # keep the GPU busy until the sampler reports (nvidia-smi starts in ~0.1-0.5 s)
        t_soak = time.perf_counter()
        i = 0
        while (len(clk.lines) < 3 and time.perf_counter() - t_soak < 5.0) or i < args.warmup:
            g_step[i % nsets].replay()
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize(dev)
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            g_step[i % nsets].replay()
        t_end.record(stream)
        barrier()
        for i in range(args.steps):
            k = i % nsets
            g_mask[k].replay()
            evs[i][0].record(stream)
            g_attn[k].replay()
            evs[i][1].record(stream)
            g_acc[k].replay()
            evs[i][2].record(stream)
        barrier()
        # a few more samples under load after the timed region
        t_tail = time.perf_counter()
        n0 = len(clk.lines)
        i = 0
        while len(clk.lines) < n0 + 2 and time.perf_counter() - t_tail < 2.0:
            g_step[i % nsets].replay()
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
    ms_local = t_start.elapsed_time(t_end) / args.steps

    # launch-amortised: 100 consecutive steps (rotating input sets) captured
    # as one CUDA graph, replayed after one warm-up replay
    g100 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g100, stream=cap):
        for i in range(100):
            step(sets[i % nsets])
    g100.replay()
    barrier()
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(3):
        g100.replay()
    h1.record(stream)
    barrier()
    ms100_local = h0.elapsed_time(h1) / 300
    attn_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    acc_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps

    # ---- KV commit of the accepted path (one layer), timed on its own after
    # the step: it rewrites tree rows of the cache in place, which later
    # replays of the step read as ordinary (finite) K/V
    commit_out = {}

    def commit_call(s):
        sv.kv_commit(s["k"], s["v"], s["page_table"], s["seq_lens"], acc_out["path"],
                     acc_out["accept_len"], outputs=commit_out)

    commit_call(sets[0])
    barrier()
    g_commit = [capture(commit_call, s) for s in sets]
    barrier()
    cevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        cevs[i][0].record(stream)
        g_commit[i % nsets].replay()
        cevs[i][1].record(stream)
    barrier()
    commit_ms = sum(e[0].elapsed_time(e[1]) for e in cevs) / args.steps
    assert int(commit_out["status"].abs().sum()) == 0

    # ---- the target-only acceptance variants on the same inputs, each timed
    # on its own (greedy argmax matching; one-hot candidate sampling)
    var_out = {"greedy": {}, "onehot": {}}

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
    e2rows = [torch.randn((B, 1 if r == 0 else e2k, w.V), generator=e2gen, device=dev) * 2.0
              for r in range(e2rounds)]
    e2roots = torch.zeros((B,), dtype=torch.int32, device=dev)
    e2cap = 1 + e2k + (e2rounds - 1) * e2k * e2k
    e2pool = sv.eagle2_pool(e2roots, e2cap)
    e2f0 = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    e2fr = [torch.empty((B, e2k), dtype=torch.int32, device=dev) for _ in range(e2rounds)]

    def eagle2_call(s):
        sv.eagle2_init(e2pool, e2roots)
        f = e2f0
        for r in range(e2rounds):
            f = sv.eagle2_expand(e2pool, e2rows[r], f, e2k, next_frontier=e2fr[r])
        return sv.eagle2_finalize(e2pool, N, outputs=e2out)

    # the walk on bf16 copies of the logits (one input set: larger than L2)
    bf_logits = {k: sets[0][k].to(torch.bfloat16) for k in ("target", "draft")}
    var_out["bf16"] = {}

    def bf16_call(s):
        sv.spec_accept(bf_logits["target"], bf_logits["draft"], s["tokens"], s["parent"],
                       s["u_accept"], s["u_bonus"], outputs=var_out["bf16"])

    var_out["greedy_bf16"] = {}
    var_out["onehot_bf16"] = {}

    def greedy_bf16_call(s):
        sv.spec_accept_greedy(bf_logits["target"], s["tokens"], s["parent"],
                              outputs=var_out["greedy_bf16"])

    def onehot_bf16_call(s):
        sv.spec_accept_onehot(bf_logits["target"], s["tokens"], s["parent"], s["u_accept"],
                              s["u_bonus"], outputs=var_out["onehot_bf16"])

    e2out = {}
    var_ms = {}
    for name, fn in (("greedy", greedy_call), ("onehot", onehot_call), ("eagle2", eagle2_call),
                     ("bf16", bf16_call), ("greedy_bf16", greedy_bf16_call),
                     ("onehot_bf16", onehot_bf16_call)):
        fn(sets[0])
        barrier()
        graphs = [capture(fn, s) for s in sets]
        barrier()
        vev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            vev[i][0].record(stream)
            graphs[i % nsets].replay()
            vev[i][1].record(stream)
        barrier()
        var_ms[name] = sum(e[0].elapsed_time(e[1]) for e in vev) / args.steps
        if name != "eagle2":
            assert int(var_out[name]["status"].abs().sum()) == 0
    assert int(e2out["n_out"].min()) == min(N, e2cap)

    def rmax(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def rsum(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    ms, value = aggregate(ms_local, B * N, world, rmax, rsum)
    ms100 = rmax(ms100_local)

    # ---- end to end through the public API from pinned host buffers. The
    # inputs of a step sit in one pinned host buffer and travel in one copy
    # into one of two device buffers whose slices the step's tensors view; a
    # side stream copies step i + 1 while step i runs (double buffering), and
    # every step's outputs come back to pinned host memory.
    offs, total = {}, 0
    for k, v in base.items():
        nbytes = v.numel() * v.element_size()
        offs[k] = (total, nbytes, v.shape, v.dtype)
        total += (nbytes + 255) & ~255
    host_in = torch.empty((total,), dtype=torch.uint8).pin_memory()
    for k, (o, nbytes, _, _) in offs.items():
        host_in[o:o + nbytes].copy_(base[k].reshape(-1).view(torch.uint8).cpu())
    dbufs = [torch.empty((total,), dtype=torch.uint8, device=dev) for _ in range(2)]
    dsets = [{k: buf[o:o + nbytes].view(dt).view(shape)
              for k, (o, nbytes, shape, dt) in offs.items()} for buf in dbufs]
    h2d = sum(nbytes for _, nbytes, _, _ in offs.values())
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    res_h = {k: torch.empty((B, N) if k in ("path", "out_tokens") else (B,),
                            dtype=torch.int32).pin_memory()
             for k in ("accept_len", "path", "out_tokens", "status")}
    d2h = out_h.numel() * out_h.element_size() + sum(t.numel() * 4 for t in res_h.values())
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
            step(dsets[j])
            used[j].record(stream)
            out_h.copy_(out, non_blocking=True)
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

    # ---- checks that the timed work produced valid results
    torch.cuda.synchronize(dev)
    assert int(astat.abs().sum()) == 0 and int(acc_out["status"].abs().sum()) == 0
    assert bool(torch.isfinite(out.float()).all())

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    attn_gbs = nb["attn_bytes"] / (attn_ms / 1e3) / 1e9
    # the walk reads only the rows of the nodes it visits (every input set is a
    # copy of the same data, so the last walk stands for all)
    acc_bytes = walk_bytes(w, inp.parent, acc_out["path"].cpu().numpy(),
                           acc_out["accept_len"].cpu().numpy())
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
    acc_ws_need = sv.spec_accept_workspace_size(B, N, w.V)
    launches_per_step = 1 + 1 + (1 if ws_need > 0 else 0) + (2 if acc_ws_need > 0 else 1)
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
            "workload": w.name, "B": B, "N": N, "context": w.L if w.L_hi is None else
            f"U[{w.L},{w.L_hi}]", "Hq": Hq, "Hkv": w.Hkv, "head_dim": D, "vocab": w.V,
            "page_size": inp.page_size, "tree": w.tree,
            "l2": f"inputs rotate over {nsets} copies ({nsets * step_bytes / 1e6:.0f} MB > "
                  f"L2 {l2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": "one CUDA graph per step (masks, attention, acceptance)",
            "e2e_copies": "one packed pinned host-to-device copy per step, issued one step "
                          "ahead on a side stream; outputs read back every step",
        },
        "accept_steps_per_s": rsum(B) / (ms / 1e3),
        "graph_100_steps": {"ms_per_step": ms100, "value": rsum(B * N) / (ms100 / 1e3),
                            "note": "100 steps captured as one CUDA graph"},
        "kernels": {
            "tree_verify_attn": {"ms": attn_ms, "bytes": nb["attn_bytes"], "gbs": attn_gbs,
                                 "frac_of_hbm": attn_gbs / peak},
            "spec_accept": {"ms": acc_ms, "bytes": acc_bytes, "gbs": acc_gbs,
                            "frac_of_hbm": acc_gbs / peak,
                            "bytes_all_rows": nb["accept_bytes"],
                            "bytes_note": "rows of the visited nodes; bytes_all_rows counts "
                                          "every row a walk could test"},
            "kv_commit": {"ms": commit_ms, "bytes": commit_bytes, "gbs": commit_gbs,
                          "frac_of_hbm": commit_gbs / peak, "rows_moved": rows_moved,
                          "bytes_note": "K and V rows of accepted nodes not yet in place, "
                                        "read and written, one layer"},
            **var_kernels,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "tree_verify_attn",
            "achieved": attn_gbs,
            "peak": peak,
            "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
            "unit": "GB/s",
            "frac": attn_gbs / peak,
            "traffic": committed_traffic(w.name, "speculative_decoding_tree_03_gb300/csrc/attn_tc.cu"),
        },
        "e2e": {"value": e2e_value, "unit": "nodes/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        per_step, sample, cores = time_oracle(inp)
        line["cpu_baseline"] = {"value": B * N / per_step, "unit": "nodes/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
        if idx <= 2:
            # the small workloads are also timed on one core
            import oracle
            per1, sample1, _ = time_oracle(inp, budget_s=10.0, max_steps=5, threads=1)
            oracle.set_threads(cores)
            line["cpu_baseline"]["single_thread"] = {"value": B * N / per1, "unit": "nodes/s",
                                                     "cores": 1, "sample": sample1}
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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    idx, w = workload_by_name(args.workload)
    if args.impl == "reference":
        run_reference(args, w, idx)
    else:
        run_ours(args, w, idx)


if __name__ == "__main__":
    main()
