"""Seeded synthetic inputs shaped like the tree-verification workloads.

This module only draws random numbers and builds draft trees. It holds none of
the verification arithmetic (ancestor masks, tree attention, acceptance): the
CUDA path and the CPU oracle both read what it produces, and neither is
imported here.

Every random tensor comes from its own numpy PCG64 stream keyed by
``SeedSequence([seed, tag, ...indices])``. A chunk (one sequence's K for one KV
head, one logits row, ...) can therefore be regenerated alone, which lets the
full-size parity tests rebuild only the slices the oracle samples.

Workload shapes follow the problem statement of tree verification in
"EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解
(parts A, B, E.1-E.3): a draft tree flattened in BFS order with a parent[]
array, a cached KV prefix, and per-node target / draft logits. The pages'
benchmarks (MT-bench, ShareGPT, SpecBench, ...) are not used; these seeded
tensors stand in for them.
"""

from __future__ import annotations

import math
import os
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# Stream tags: one per kind of random tensor.
TAG_Q, TAG_K, TAG_V, TAG_TGT, TAG_NOISE = 1, 2, 3, 4, 5
TAG_UACC, TAG_UBON, TAG_PAGES, TAG_LENS, TAG_ROOT, TAG_DRAW = 6, 7, 8, 9, 10, 11


def rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, key)])))


# ----------------------------------------------------------------------------
# bf16 storage helpers (round-to-nearest-even), plain bit manipulation.
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even. No NaNs expected."""
    u = np.ascontiguousarray(x, dtype=np.float32).copy().view(np.uint32)
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    u += r
    u += np.uint32(0x7FFF)
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exact."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_chunk(seed: int, key: tuple, shape, bf16: bool) -> np.ndarray:
    """N(0,1) draws for one keyed chunk: float32, or bf16 bits if ``bf16``."""
    x = rng(seed, *key).standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(shape)
    return f32_to_bf16_bits(x) if bf16 else x


# ----------------------------------------------------------------------------
# Workload table
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int                      # tree nodes including the root
    tree: str                   # "chain" | "binary" | "eagle2"
    L: int                      # prefix length (or lower bound when L_hi is set)
    Hq: int
    Hkv: int
    D: int
    dtype: str                  # "f32" | "bf16" (q, K, V, attention output)
    V: int                      # vocabulary
    target_sigma: float
    draft_sigma: float
    L_hi: Optional[int] = None  # per-sequence prefix lengths uniform in [L, L_hi]
    page_size: int = 0          # 0: contiguous cache, one page per sequence
    binary_depth: int = 0
    eagle2_topk: int = 8
    eagle2_rounds: int = 6
    desc: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


WORKLOADS = [
    Workload("tiny_chain", B=1, N=4, tree="chain", L=128, Hq=4, Hkv=4, D=64, dtype="f32",
             V=1000, target_sigma=2.0, draft_sigma=1.0,
             desc="chain of 4 nodes, fp32, context 128, 4/4 heads, head_dim 64, vocab 1000"),
    Workload("binary_tree_8b", B=1, N=31, tree="binary", binary_depth=4, L=2048, Hq=32, Hkv=8, D=128,
             dtype="bf16", V=32000, target_sigma=3.0, draft_sigma=1.5,
             desc="depth-4 binary tree (31 nodes), batch 1, context 2048, 32/8 heads, d128, vocab 32000"),
    Workload("eagle2_tree_8b", B=4, N=60, tree="eagle2", L=8192, Hq=32, Hkv=8, D=128, dtype="bf16",
             V=128256, target_sigma=3.0, draft_sigma=1.0,
             desc="EAGLE-2 dynamic tree (60 nodes, depth<=6, top-8), batch 4, context 8192, vocab 128256"),
    Workload("paged_block_chain", B=16, N=16, tree="chain", L=1024, L_hi=4096, Hq=32, Hkv=8, D=128,
             dtype="bf16", V=151936, target_sigma=3.0, draft_sigma=2.0, page_size=16,
             desc="16-node chain, batch 16, context U[1024,4096], paged 16, vocab 151936"),
    Workload("serving_70b", B=64, N=31, tree="binary", binary_depth=4, L=32768, Hq=64, Hkv=8, D=128,
             dtype="bf16", V=128256, target_sigma=3.0, draft_sigma=1.5, page_size=16,
             desc="31-node binary tree per sequence, batch 64, context 32768, 64/8 heads, paged 16"),
]


def default_seed(idx: int) -> int:
    return 1000 + idx


# ----------------------------------------------------------------------------
# Trees
# ----------------------------------------------------------------------------

def chain_parent(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def binary_tree_parent(depth: int) -> np.ndarray:
    n = 2 ** (depth + 1) - 1
    p = (np.arange(n, dtype=np.int64) - 1) // 2
    p[0] = -1
    return p.astype(np.int32)


def draft_probs(row: np.ndarray) -> np.ndarray:
    """Draft softmax of one logits row, used only to pick tree tokens."""
    r = row.astype(np.float64)
    e = np.exp(r - r.max())
    return e / e.sum()


def topk_tokens(probs: np.ndarray, k: int) -> np.ndarray:
    """Top-k token ids by probability, descending; ties go to the lower id."""
    ids = np.arange(probs.shape[0])
    order = np.lexsort((ids, -probs))
    return order[:k]


def eagle2_expand_step(frontier_values, child_conf, k):
    """One EAGLE-2 expansion step on plain numbers.

    The k frontier nodes with the largest value are expanded; each child's value
    is its parent's value times its own draft confidence, and the new frontier
    is ordered by value. This is the step worked through in "EAGLE 演化史",
    § E.3 (frontier {0.95, 0.6, 0.3, 0.05}, k=2).

    Returns (expanded parent positions, children values in creation order,
    new frontier values sorted descending).
    """
    fv = np.asarray(frontier_values, dtype=np.float64)
    sel = np.lexsort((np.arange(fv.size), -fv))[:k]
    children = []
    for j, pos in enumerate(sel):
        for c in child_conf[j]:
            children.append(fv[pos] * c)
    children = np.array(children)
    return sel, children, np.sort(children)[::-1]


@dataclass
class _Node:
    cid: int
    parent: int        # creation id of the parent, -1 for the root
    depth: int
    value: float
    token: int
    conf: float


def build_eagle2_tree(draft_row_of, root_token: int, topk: int, rounds: int, n_nodes: int):
    """EAGLE-2 expand-then-rerank tree construction.

    ``draft_row_of(cid)`` returns the draft logits row at the node with that
    creation id. Expansion ("EAGLE 演化史" § E.2; "The EAGLE Family", EAGLE-2):
    round 1 expands the root into its top-k draft tokens; each later round
    expands the top-k of the previous round's new nodes (by value, ties to the
    lower creation id) into their top-k children. A node's value is the product
    of draft confidences on its root path, the confidence being the draft
    probability of the node's own token. Rerank keeps the root plus the
    n_nodes-1 best by (value desc, depth asc, creation id asc), which is a
    connected subtree, and renumbers it in BFS order by (depth, parent's new
    index, value desc, creation id).

    Returns (parent[n_nodes] int32 in BFS numbering, creation ids in BFS order,
    tokens in BFS order, values in BFS order).
    """
    nodes = [_Node(0, -1, 0, 1.0, int(root_token), 1.0)]

    def expand(nd: _Node):
        q = draft_probs(draft_row_of(nd.cid))
        out = []
        for t in topk_tokens(q, topk):
            c = float(q[t])
            child = _Node(len(nodes), nd.cid, nd.depth + 1, nd.value * c, int(t), c)
            nodes.append(child)
            out.append(child)
        return out

    new = expand(nodes[0])
    for _ in range(2, rounds + 1):
        sel = sorted(new, key=lambda n: (-n.value, n.cid))[:topk]
        new = [c for nd in sel for c in expand(nd)]

    keep = sorted(nodes[1:], key=lambda n: (-n.value, n.depth, n.cid))[: n_nodes - 1]
    kept = {0} | {n.cid for n in keep}
    for n in keep:
        assert n.parent in kept, "top-N by path value must be a connected subtree"

    by_cid = {n.cid: n for n in nodes}
    order = [0]
    new_index = {0: 0}
    max_depth = max(n.depth for n in keep) if keep else 0
    for d in range(1, max_depth + 1):
        level = [n for n in keep if n.depth == d]
        level.sort(key=lambda n: (new_index[n.parent], -n.value, n.cid))
        for n in level:
            new_index[n.cid] = len(order)
            order.append(n.cid)
    parent = np.array([-1] + [new_index[by_cid[c].parent] for c in order[1:]], dtype=np.int32)
    tokens = np.array([by_cid[c].token for c in order], dtype=np.int32)
    values = np.array([by_cid[c].value for c in order], dtype=np.float64)
    return parent, np.array(order, dtype=np.int64), tokens, values


# ----------------------------------------------------------------------------
# Logits rows
# ----------------------------------------------------------------------------

def target_row(seed, b, rowkey, V, sigma):
    return (sigma * rng(seed, TAG_TGT, b, rowkey).standard_normal(V, dtype=np.float32)).astype(np.float32)


def draft_row(seed, b, rowkey, V, sigma_t, sigma_d):
    noise = sigma_d * rng(seed, TAG_NOISE, b, rowkey).standard_normal(V, dtype=np.float32)
    return (target_row(seed, b, rowkey, V, sigma_t) + noise.astype(np.float32)).astype(np.float32)


def make_tree(w: Workload, seed: int, b: int):
    """Tree of sequence b: (parent[N], row keys[N], tokens[N])."""
    root = int(rng(seed, TAG_ROOT, b).integers(0, w.V))
    if w.tree == "chain":
        parent = chain_parent(w.N)
        keys = np.arange(w.N)
        tokens = np.empty(w.N, dtype=np.int32)
        tokens[0] = root
        for i in range(1, w.N):
            q = draft_probs(draft_row(seed, b, i - 1, w.V, w.target_sigma, w.draft_sigma))
            u = rng(seed, TAG_DRAW, b, i).random()
            cdf = np.cumsum(q)
            tokens[i] = min(int(np.searchsorted(cdf, u * cdf[-1], side="right")), w.V - 1)
        return parent, keys, tokens
    if w.tree == "binary":
        parent = binary_tree_parent(w.binary_depth)
        assert parent.size == w.N
        keys = np.arange(w.N)
        tokens = np.empty(w.N, dtype=np.int32)
        tokens[0] = root
        for j in range(w.N):
            kids = [c for c in (2 * j + 1, 2 * j + 2) if c < w.N]
            if not kids:
                continue
            q = draft_probs(draft_row(seed, b, j, w.V, w.target_sigma, w.draft_sigma))
            top = topk_tokens(q, len(kids))
            for c, t in zip(kids, top):
                tokens[c] = t
        return parent, keys, tokens
    if w.tree == "eagle2":
        cache = {}

        def row_of(cid):
            if cid not in cache:
                cache[cid] = draft_row(seed, b, cid, w.V, w.target_sigma, w.draft_sigma)
            return cache[cid]

        parent, keys, tokens, _ = build_eagle2_tree(row_of, root, w.eagle2_topk, w.eagle2_rounds, w.N)
        return parent, keys, tokens
    raise ValueError(w.tree)


# ----------------------------------------------------------------------------
# KV cache
# ----------------------------------------------------------------------------

def prefix_lengths(w: Workload, seed: int) -> np.ndarray:
    if w.L_hi is None:
        return np.full(w.B, w.L, dtype=np.int32)
    return rng(seed, TAG_LENS).integers(w.L, w.L_hi + 1, size=w.B).astype(np.int32)


def logical_kv(w: Workload, seed: int, b: int, g: int, T: int):
    """K and V of sequence b, KV head g, logical tokens [0, T): arrays [T, D] (f32 or bf16 bits)."""
    bf = w.dtype == "bf16"
    return (normal_chunk(seed, (TAG_K, b, g), (T, w.D), bf),
            normal_chunk(seed, (TAG_V, b, g), (T, w.D), bf))


def page_layout(w: Workload, seed: int, seq_lens: np.ndarray):
    """(page_size, num_pages, page_table[B, max_pages]) for the workload's cache.

    Contiguous caches use one page per sequence whose size is the longest
    sequence rounded up to 128 tokens. Paged caches use ``w.page_size`` tokens
    per page and a seeded random permutation of page ids; unused table entries
    are -1.
    """
    T = seq_lens.astype(np.int64) + w.N
    if w.page_size == 0:
        ps = int(-(-int(T.max()) // 128) * 128)
        table = np.arange(w.B, dtype=np.int32).reshape(w.B, 1)
        return ps, w.B, table
    ps = w.page_size
    n = -(-T // ps)
    P = int(n.sum())
    perm = rng(seed, TAG_PAGES).permutation(P).astype(np.int32)
    table = np.full((w.B, int(n.max())), -1, dtype=np.int32)
    off = 0
    for b in range(w.B):
        table[b, : n[b]] = perm[off: off + n[b]]
        off += int(n[b])
    return ps, P, table


def _kv_chunk(args):
    w, seed, b, g, T = args
    return b, g, logical_kv(w, seed, b, g, T)


def build_kv_cache(w: Workload, seed: int, seq_lens, page_size, num_pages, table, workers: int = 0):
    """Paged K and V caches [num_pages, page_size, Hkv, D] (float32 or bf16 bits).

    Large caches draw their (sequence, KV head) chunks in a pool of spawned
    processes; this process scatters each returned chunk into the pages."""
    dt = np.uint16 if w.dtype == "bf16" else np.float32
    shape = (num_pages, page_size, w.Hkv, w.D)
    T_all = seq_lens.astype(np.int64) + w.N
    kc = np.zeros(shape, dtype=dt)
    vc = np.zeros(shape, dtype=dt)
    kflat = kc.reshape(num_pages * page_size, w.Hkv, w.D)
    vflat = vc.reshape(num_pages * page_size, w.Hkv, w.D)
    slot_of = {}

    def slots(b):
        if b not in slot_of:
            t = np.arange(int(T_all[b]))
            slot_of[b] = table[b, t // page_size].astype(np.int64) * page_size + t % page_size
        return slot_of[b]

    jobs = [(w, seed, b, g, int(T_all[b])) for b in range(w.B) for g in range(w.Hkv)]
    nbytes = int(np.prod(shape)) * np.dtype(dt).itemsize
    if workers <= 1 or nbytes < (256 << 20):
        results = map(_kv_chunk, jobs)
        for b, g, (k, v) in results:
            kflat[slots(b), g, :] = k
            vflat[slots(b), g, :] = v
        return kc, vc
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(workers) as pool:
        for b, g, (k, v) in pool.imap_unordered(_kv_chunk, jobs, chunksize=2):
            kflat[slots(b), g, :] = k
            vflat[slots(b), g, :] = v
    return kc, vc


# ----------------------------------------------------------------------------
# Whole workload
# ----------------------------------------------------------------------------

@dataclass
class Inputs:
    w: Workload
    seed: int
    seq_lens: np.ndarray          # [B] int32, prefix length (tree excluded)
    parent: np.ndarray            # [B, N] int32
    tokens: np.ndarray            # [B, N] int32
    row_keys: np.ndarray          # [B, N] int64 (stream keys of each node's logits rows)
    q: np.ndarray                 # [B, N, Hq, D] float32 or bf16 bits
    page_size: int
    num_pages: int
    page_table: np.ndarray        # [B, max_pages] int32
    k_cache: Optional[np.ndarray]  # [num_pages, page_size, Hkv, D]
    v_cache: Optional[np.ndarray]
    target: Optional[np.ndarray]  # [B, N, V] float32
    draft: Optional[np.ndarray]   # [B, N, V] float32
    u_accept: np.ndarray          # [B, N] float32 in [0, 1)
    u_bonus: np.ndarray           # [B] float32 in [0, 1)
    extra: dict = field(default_factory=dict)


def _logits_rows(w, seed, b, keys):
    t = np.stack([target_row(seed, b, int(k), w.V, w.target_sigma) for k in keys])
    d = np.stack([draft_row(seed, b, int(k), w.V, w.target_sigma, w.draft_sigma) for k in keys])
    return t, d


def _sequence_job(args):
    """Tree and (optionally) logits rows of one sequence."""
    w, seed, b, with_logits = args
    parent, keys, tokens = make_tree(w, seed, b)
    rows = _logits_rows(w, seed, b, keys) if with_logits else None
    return parent, keys, tokens, rows


def make_inputs(w: Workload, seed: int, with_kv: bool = True, with_logits: bool = True,
                workers: Optional[int] = None) -> Inputs:
    """All inputs of one workload, as host arrays. Large batches build their
    sequences' trees and logits in a pool of spawned processes; every value
    comes from its own keyed stream, so the result does not depend on it."""
    if workers is None:
        workers = min(16, os.cpu_count() or 1)
    seq_lens = prefix_lengths(w, seed)
    parent = np.empty((w.B, w.N), dtype=np.int32)
    tokens = np.empty((w.B, w.N), dtype=np.int32)
    keys = np.empty((w.B, w.N), dtype=np.int64)
    tgt = dft = None
    if with_logits:
        tgt = np.empty((w.B, w.N, w.V), dtype=np.float32)
        dft = np.empty((w.B, w.N, w.V), dtype=np.float32)
    jobs = [(w, seed, b, with_logits) for b in range(w.B)]
    if workers > 1 and w.B >= 8 and w.N * w.V >= (1 << 20):
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(min(workers, w.B)) as pool:
            results = pool.map(_sequence_job, jobs, chunksize=1)
    else:
        results = map(_sequence_job, jobs)
    for b, (pa, ke, to, rows) in enumerate(results):
        parent[b], keys[b], tokens[b] = pa, ke, to
        if with_logits:
            tgt[b], dft[b] = rows
    bf = w.dtype == "bf16"
    q = np.stack([normal_chunk(seed, (TAG_Q, b), (w.N, w.Hq, w.D), bf) for b in range(w.B)])
    ps, P, table = page_layout(w, seed, seq_lens)
    kc = vc = None
    if with_kv:
        kc, vc = build_kv_cache(w, seed, seq_lens, ps, P, table, workers=workers)
    u_acc = np.stack([rng(seed, TAG_UACC, b).random(w.N, dtype=np.float32) for b in range(w.B)])
    u_bon = np.array([rng(seed, TAG_UBON, b).random(dtype=np.float32) for b in range(w.B)],
                     dtype=np.float32)
    return Inputs(w, seed, seq_lens, parent, tokens, keys, q, ps, P, table, kc, vc, tgt, dft,
                  u_acc, u_bon)


def logits_of(inp: Inputs, b: int):
    """Target and draft logits [N, V] of sequence b, regenerated from their streams."""
    return _logits_rows(inp.w, inp.seed, b, inp.row_keys[b])


def algorithmic_bytes(w: Workload, seq_lens: np.ndarray, parent: np.ndarray) -> dict:
    """Bytes one call must move at minimum, per kernel.

    Attention: K and V of the prefix and tree tokens once per (sequence, KV
    head), q read and output written once, the ancestor masks read once.
    Acceptance: the target row of every node and the draft row of every node
    that has children, fp32, each read once.
    """
    es = 2 if w.dtype == "bf16" else 4
    T = seq_lens.astype(np.int64) + w.N
    kv = int(T.sum()) * w.Hkv * w.D * es * 2
    qo = w.B * w.N * w.Hq * w.D * es * 2
    mask = w.B * w.N * 8
    attn = kv + qo + mask
    internal = 0
    for b in range(parent.shape[0]):
        internal += len(set(int(x) for x in parent[b, 1:]))
    accept = (w.B * w.N + internal) * w.V * 4
    flops = 4 * int(T.sum()) * w.N * w.Hq * w.D
    return {"attn_bytes": attn, "accept_bytes": accept, "attn_flops": flops,
            "internal_rows": internal}

