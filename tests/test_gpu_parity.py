"""GPU parity: every kernel through the C ABI against the fp64 oracle.

Masks, accepted paths, accepted lengths and tokens must match bit for bit
(near ties aside, under the error model in gpu_common); acceptance ratios
within 1e-5 relative at first tests; attention outputs within max-abs 2e-2
(bf16 inputs and output) or 1e-5 (fp32), lse within 2e-3 (bf16) or 1e-5.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (bf16_tensor, compare_accept, device_inputs, oracle_attention,
                        as_f32)
from synth import WORKLOADS, make_inputs, binary_tree_parent, chain_parent
from synth.gen import Workload, f32_to_bf16_bits, bf16_bits_to_f32

pytestmark = pytest.mark.gpu

BF16_OUT_TOL = 2e-2
BF16_LSE_TOL = 2e-3
F32_TOL = 1e-5


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


def _np(t):
    return t.detach().cpu().numpy()


# the two bf16 attention kernels: 1 = chunks of a unit merged inside a
# thread-block cluster, 2 = one persistent CTA per SM over an equal share of
# all units' tiles, split units merged through the workspace
KERNELS = [1, 2]


@pytest.fixture(params=KERNELS, ids=["cluster", "persistent"])
def attn_kernel(sv, request):
    lib = sv.load_library()
    assert lib.svf_debug_set_attn_kernel(request.param) == 0
    yield request.param
    lib.svf_debug_set_attn_kernel(0)


# ---------------------------------------------------------------------------
# tree_mask_build
# ---------------------------------------------------------------------------

def _random_parents(rng, B, N):
    return np.stack([np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)
                     for _ in range(B)])


@pytest.mark.parametrize("N", [1, 2, 7, 31, 60, 64, 65, 200, 1024])
def test_mask_matches_oracle(sv, N):
    rng = np.random.default_rng(N)
    parent = _random_parents(rng, 5, N)
    parent[1] = np.arange(-1, N - 1)  # a chain
    anc, depth, status = sv.tree_mask_build(torch.from_numpy(parent).cuda())
    oa, od, os_ = oracle.tree_mask(parent)
    assert (_np(anc).view(np.uint64) == oa).all()
    assert (_np(depth) == od).all() and (_np(status) == os_).all()


def test_mask_invalid_trees(sv):
    bad = np.array([[0, 0, 1, 2], [-1, 1, 0, 0], [-1, 0, 5, 1], [-1, 0, 1, 1]], np.int32)
    anc, depth, status = sv.tree_mask_build(torch.from_numpy(bad).cuda())
    oa, od, os_ = oracle.tree_mask(bad)
    assert _np(status).tolist() == [1, 1, 1, 0]
    assert (_np(anc).view(np.uint64) == oa).all() and (_np(depth) == od).all()


def test_empty_batch_is_a_no_op(sv):
    lib = sv.load_library()
    assert lib.svf_tree_mask_build(None, 0, 4, None, None, None, None) == 0
    assert lib.svf_spec_accept(None, None, None, None, None, None, 0, 4, 10, None, None, None,
                               None, None, 0, None, None) == 0


# ---------------------------------------------------------------------------
# tree_verify_attn
# ---------------------------------------------------------------------------

def _attn_case(seed, B, N, parent, lens, Hq, Hkv, D, dtype, page_size, extra_pages=3):
    """Random attention inputs with a paged (or contiguous) cache."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    T = lens.astype(np.int64) + N
    if page_size == 0:
        ps = int(-(-int(T.max()) // 128) * 128)
        n = np.ones(B, np.int64)
    else:
        ps = page_size
        n = -(-T // ps)
    P = int(n.sum()) + extra_pages
    perm = rng.permutation(P).astype(np.int32)
    table = np.full((B, int(n.max())), -1, np.int32)
    off = 0
    for b in range(B):
        table[b, : n[b]] = perm[off: off + n[b]]
        off += int(n[b])
    q = rng.standard_normal((B, N, Hq, D)).astype(np.float32)
    kc = rng.standard_normal((P, ps, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((P, ps, Hkv, D)).astype(np.float32)
    if dtype == "bf16":
        q, kc, vc = (bf16_bits_to_f32(f32_to_bf16_bits(x)) for x in (q, kc, vc))
    # logical K/V for the oracle, read through the page table
    Tcap = int(T.max())
    K = np.zeros((B, Tcap, Hkv, D), np.float32)
    V = np.zeros_like(K)
    for b in range(B):
        t = np.arange(T[b])
        pages = table[b, t // ps]
        K[b, : T[b]] = kc[pages, t % ps]
        V[b, : T[b]] = vc[pages, t % ps]
    return dict(q=q, kc=kc, vc=vc, table=table, lens=lens, parent=np.asarray(parent, np.int32),
                K=K, V=V, ps=ps, P=P)


def _run_attn(sv, c, dtype, poison_tail=False):
    dev = "cuda"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.from_numpy(c["q"]).to(dev).to(tdt)
    kc = torch.from_numpy(c["kc"]).to(dev).to(tdt)
    vc = torch.from_numpy(c["vc"]).to(dev).to(tdt)
    if poison_tail:
        # slots past each sequence's end inside its last page hold NaN
        B = c["q"].shape[0]
        N = c["q"].shape[1]
        for b in range(B):
            T = int(c["lens"][b]) + N
            last = int(c["table"][b, (T - 1) // c["ps"]])
            s0 = T % c["ps"]
            if s0:
                kc[last, s0:] = float("nan")
                vc[last, s0:] = float("nan")
    parent = torch.from_numpy(c["parent"]).to(dev)
    anc, _, _ = sv.tree_mask_build(parent)
    out, lse, status = sv.tree_verify_attn(q, kc, vc, torch.from_numpy(c["table"]).to(dev),
                                           torch.from_numpy(c["lens"]).to(dev), anc)
    torch.cuda.synchronize()
    return _np(out.float()), _np(lse), _np(status)


CASES = [
    # name, seed, B, parent, lens, Hq, Hkv, D, dtype, page_size
    ("worked_tree_contig", 1, 2, "worked", [300, 129], 8, 2, 128, "bf16", 0),
    ("binary31_paged16_g8", 2, 3, "binary4", [1000, 17, 385], 16, 2, 128, "bf16", 16),
    ("random60_paged32_rowblocks", 3, 2, "random60", [700, 250], 8, 1, 128, "bf16", 32),
    ("single_node_no_prefix", 4, 2, "single", [0, 5], 4, 4, 128, "bf16", 128),
    ("tree_crosses_tile", 5, 2, "random64", [100, 64], 8, 2, 128, "bf16", 64),
    ("chain16_paged256", 6, 3, "chain16", [2000, 1, 511], 32, 8, 128, "bf16", 256),
    ("g1_many_heads", 7, 1, "binary3", [900], 8, 8, 128, "bf16", 16),
    ("fp32_d64", 8, 2, "worked", [200, 3], 4, 4, 64, "f32", 0),
    ("fp32_d128_paged", 9, 2, "binary3", [150, 40], 8, 2, 128, "f32", 16),
    # 80 (sequence, KV head) units, lengths from 7 to 2000 tokens
    ("bf16_mixed_lengths", 13, 10, "chain16",
     [40, 900, 120, 2000, 333, 64, 1500, 7, 250, 1100], 32, 8, 128, "bf16", 16),
]


def _parent_of(kind, B, rng):
    if kind == "worked":
        p = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
    elif kind == "binary4":
        p = binary_tree_parent(4)
    elif kind == "binary3":
        p = binary_tree_parent(3)
    elif kind == "single":
        p = np.array([-1], np.int32)
    elif kind == "chain16":
        p = chain_parent(16)
    elif kind.startswith("random"):
        N = int(kind[6:])
        return _random_parents(rng, B, N)
    return np.broadcast_to(p, (B, p.size)).copy()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_small_cases(sv, attn_kernel, case):
    name, seed, B, pk, lens, Hq, Hkv, D, dtype, ps = case
    parent = _parent_of(pk, B, np.random.default_rng(seed + 100))
    N = parent.shape[1]
    c = _attn_case(seed, B, N, parent, lens, Hq, Hkv, D, dtype, ps)
    out, lse, status = _run_attn(sv, c, dtype)
    assert (status == 0).all()
    o_ref, l_ref = oracle.tree_attn(c["q"], c["K"], c["V"], c["lens"], c["parent"])
    o_ref = o_ref.reshape(out.shape)
    l_ref = l_ref.reshape(lse.shape)
    tol_o = BF16_OUT_TOL if dtype == "bf16" else F32_TOL
    tol_l = BF16_LSE_TOL if dtype == "bf16" else F32_TOL
    err_o = np.abs(out - o_ref).max()
    err_l = np.abs(lse - l_ref).max()
    print(f"{name} kernel {attn_kernel}: max|out-ref| {err_o:.3g} max|lse-ref| {err_l:.3g}")
    assert err_l <= tol_l, err_l
    assert err_o <= tol_o, err_o


def test_attention_ignores_garbage_past_sequence_end(sv, attn_kernel):
    parent = binary_tree_parent(3)
    B = 2
    parent = np.broadcast_to(parent, (B, parent.size)).copy()
    c = _attn_case(11, B, parent.shape[1], parent, [77, 301], 8, 2, 128, "bf16", 0)
    out, lse, status = _run_attn(sv, c, "bf16", poison_tail=True)
    o_ref, _ = oracle.tree_attn(c["q"], c["K"], c["V"], c["lens"], c["parent"])
    assert np.isfinite(out).all()
    assert np.abs(out - o_ref.reshape(out.shape)).max() <= BF16_OUT_TOL


def test_attention_bad_page_and_length_status(sv, attn_kernel):
    parent = binary_tree_parent(2)
    B = 3
    parent = np.broadcast_to(parent, (B, parent.size)).copy()
    c = _attn_case(12, B, parent.shape[1], parent, [200, 90, 33], 8, 2, 128, "bf16", 16)
    c["table"][1, 2] = c["P"] + 7          # page id outside the cache
    c["lens"][2] = c["table"].shape[1] * 16  # overflows its page table
    for dtype in ("bf16", "f32"):
        out, lse, status = _run_attn(sv, c, dtype)
        assert status.tolist() == [0, 4, 8], status
        assert (out[1] == 0).all() and (out[2] == 0).all()
        o_ref, _ = oracle.tree_attn(c["q"][:1], c["K"][:1], c["V"][:1], c["lens"][:1],
                                    c["parent"][:1])
        tol = BF16_OUT_TOL if dtype == "bf16" else F32_TOL
        assert np.abs(out[0] - o_ref.reshape(out[0].shape)).max() <= tol


def test_attention_mixed_lengths_with_bad_sequences(sv, attn_kernel):
    """80 units of mixed lengths with a bad page and a bad length in the batch:
    those sequences get their status bit and zeros, the rest match."""
    parent = chain_parent(16)
    B = 10
    parent = np.broadcast_to(parent, (B, parent.size)).copy()
    lens = [40, 900, 120, 2000, 333, 64, 1500, 7, 250, 1100]
    c = _attn_case(14, B, parent.shape[1], parent, lens, 32, 8, 128, "bf16", 16)
    c["table"][3, 5] = c["P"] + 9           # page id outside the cache
    c["lens"][6] = c["table"].shape[1] * 16  # overflows its page table
    out, lse, status = _run_attn(sv, c, "bf16")
    want = [0] * B
    want[3], want[6] = 4, 8
    assert status.tolist() == want, status
    assert (out[3] == 0).all() and (out[6] == 0).all()
    good = [b for b in range(B) if want[b] == 0]
    o_ref, _ = oracle.tree_attn(c["q"][good], c["K"][good], c["V"][good], c["lens"][good],
                                c["parent"][good])
    assert np.abs(out[good] - o_ref.reshape(out[good].shape)).max() <= BF16_OUT_TOL


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_attention_workloads_full(sv, attn_kernel, idx):
    w = WORKLOADS[idx]
    inp = make_inputs(w, 1000 + idx, with_kv=True, with_logits=False)
    d = device_inputs(inp)
    anc, _, _ = sv.tree_mask_build(d["parent"])
    out, lse, status = sv.tree_verify_attn(d["q"], d["k"], d["v"], d["page_table"],
                                           d["seq_lens"], anc)
    torch.cuda.synchronize()
    assert (_np(status) == 0).all()
    o_ref, l_ref = oracle_attention(inp)
    out = _np(out.float())
    err_o = np.abs(out - o_ref.reshape(out.shape)).max()
    err_l = np.abs(_np(lse) - l_ref.reshape(lse.shape)).max()
    tol_o = BF16_OUT_TOL if w.dtype == "bf16" else F32_TOL
    tol_l = BF16_LSE_TOL if w.dtype == "bf16" else F32_TOL
    print(f"{w.name}: max|out-ref| {err_o:.3g} max|lse-ref| {err_l:.3g}")
    assert err_o <= tol_o and err_l <= tol_l


def test_attention_serving_70b_sampled(sv):
    """Full-size 70B-shaped workload (8.6 GB paged cache) in the launch shape
    the benchmark times. Every (sequence, KV head) is checked on six of its
    N*G = 248 query rows: the first and last row of each 128-row half (rows
    0, 127, 128, 247) and one more row drawn in each half. Every row merges
    all KV chunks, so every chunk boundary of every sequence is crossed. The
    oracle recomputes the rows one by one, eight sequences at a time."""
    w = WORKLOADS[4]
    G = w.Hq // w.Hkv
    inp = make_inputs(w, 1004, with_kv=True, with_logits=False)
    d = device_inputs(inp)
    anc, _, _ = sv.tree_mask_build(d["parent"])
    out, lse, status = sv.tree_verify_attn(d["q"], d["k"], d["v"], d["page_table"],
                                           d["seq_lens"], anc)
    torch.cuda.synchronize()
    assert (_np(status) == 0).all()
    out = _np(out.float())
    lse = _np(lse)
    del d
    rng = np.random.default_rng(7)
    M = w.N * G
    worst_o = worst_l = 0.0
    checked = 0
    for b0 in range(0, w.B, 8):
        bs = list(range(b0, min(w.B, b0 + 8)))
        rows = []
        for n in range(len(bs)):
            for g in range(w.Hkv):
                picks = [0, 127, 128, M - 1, int(rng.integers(1, 127)),
                         int(rng.integers(129, M - 1))]
                for R in picks:
                    rows.append((n, R // G, g * G + R % G))
        o_ref, l_ref = oracle_attention(inp, bs=bs, rows=np.array(rows))
        for r, (n, i, h) in enumerate(rows):
            b = bs[n]
            worst_o = max(worst_o, float(np.abs(out[b, i, h] - o_ref[r]).max()))
            worst_l = max(worst_l, abs(float(lse[b, i, h]) - float(l_ref[r])))
        checked += len(rows)
    print(f"serving_70b: {checked} rows, max|out-ref| {worst_o:.3g} max|lse-ref| {worst_l:.3g}")
    assert checked == w.B * w.Hkv * 6
    assert worst_o <= BF16_OUT_TOL and worst_l <= BF16_LSE_TOL


# ---------------------------------------------------------------------------
# spec_accept
# ---------------------------------------------------------------------------

def _accept_gpu(sv, arrs):
    dev = "cuda"
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in arrs.items()}
    res = sv.spec_accept(t["target"], t["draft"], t["tokens"], t["parent"], t["u_accept"],
                         t["u_bonus"])
    torch.cuda.synchronize()
    return {k: (_np(v) if v is not None else None) for k, v in res.items()}


def _arrays(inp):
    return dict(target=inp.target, draft=inp.draft, tokens=inp.tokens, parent=inp.parent,
                u_accept=inp.u_accept, u_bonus=inp.u_bonus)


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_accept_workloads(sv, idx):
    w = WORKLOADS[idx]
    inp = make_inputs(w, 1000 + idx, with_kv=False, with_logits=True)
    arrs = _arrays(inp)
    gpu = _accept_gpu(sv, arrs)
    orc = oracle.spec_accept(**arrs)
    stats = compare_accept(gpu, arrs, orc)
    print(f"{w.name}: {stats} accept_len {gpu['accept_len'][:8]}")
    assert stats["ratio_rel_err_first_tests"] <= 1e-5


def _synthetic_accept(seed, B, N, V, parent, sigma=3.0, noise=1.0, iid_children=True):
    rng = np.random.default_rng(seed)
    tgt = (sigma * rng.standard_normal((B, N, V))).astype(np.float32)
    dft = (tgt + noise * rng.standard_normal((B, N, V))).astype(np.float32)
    parent = np.broadcast_to(np.asarray(parent, np.int32), (B, N)).copy()
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            j = parent[b, c]
            d = dft[b, j].astype(np.float64)
            q = np.exp(d - d.max()); q /= q.sum()
            tokens[b, c] = rng.choice(V, p=q) if iid_children else int(np.argmax(q))
    return dict(target=tgt, draft=dft, tokens=tokens, parent=parent,
                u_accept=rng.random((B, N), dtype=np.float32),
                u_bonus=rng.random(B, dtype=np.float32))


@pytest.mark.parametrize("V", [8, 37, 1000, 2049, 5003, 32000])
def test_accept_vocab_sizes(sv, V):
    """Warp-per-sequence (V <= 2048) and block-per-sequence paths, vector and
    scalar loads (V % 4)."""
    arrs = _synthetic_accept(V, 64, 7, V, [-1, 0, 0, 1, 1, 2, 2], sigma=2.0, noise=0.7)
    gpu = _accept_gpu(sv, arrs)
    orc = oracle.spec_accept(**arrs)
    stats = compare_accept(gpu, arrs, orc)
    print(V, stats)


@pytest.mark.parametrize("V", [32000, 100003])
def test_accept_many_sequences(sv, V):
    """More sequences than clusters that fit at once (vector and scalar loads)."""
    B = 100 if V == 32000 else 40
    arrs = _synthetic_accept(V + 1, B, 15, V, [-1] + [(i - 1) // 2 for i in range(1, 15)],
                             sigma=3.0, noise=1.5)
    gpu = _accept_gpu(sv, arrs)
    compare_accept(gpu, arrs, oracle.spec_accept(**arrs))


def _accept_gpu_bf16(sv, arrs):
    """The bf16 call on the logits rounded to bf16; returns the GPU results
    and the widened (exact) fp32 arrays the oracle is run on."""
    wide = dict(arrs)
    t = {}
    for k in ("target", "draft"):
        bits = f32_to_bf16_bits(np.ascontiguousarray(arrs[k], np.float32))
        wide[k] = bf16_bits_to_f32(bits)
        t[k] = bf16_tensor(bits, "cuda")
    for k in ("tokens", "parent", "u_accept", "u_bonus"):
        t[k] = torch.from_numpy(np.ascontiguousarray(arrs[k])).cuda()
    res = sv.spec_accept(t["target"], t["draft"], t["tokens"], t["parent"], t["u_accept"],
                         t["u_bonus"])
    torch.cuda.synchronize()
    return {k: (_np(v) if v is not None else None) for k, v in res.items()}, wide


@pytest.mark.parametrize("V", [8, 37, 1000, 1004, 5003, 32000, 128256])
def test_accept_bf16_logits(sv, V):
    """bf16 logits (vector and scalar loads, warp, block and cluster paths)
    against the oracle on the widened values. V = 1004: rows start on 8-byte
    but not 16-byte boundaries, so the walk's L2 prefetches are shrunk to the
    aligned interior of each slice."""
    arrs = _synthetic_accept(V + 3, 48, 7, V, [-1, 0, 0, 1, 1, 2, 2], sigma=2.0, noise=0.7)
    gpu, wide = _accept_gpu_bf16(sv, arrs)
    compare_accept(gpu, wide, oracle.spec_accept(**wide))


@pytest.mark.parametrize("idx", [1, 2])
def test_accept_bf16_workloads(sv, idx):
    w = WORKLOADS[idx]
    inp = make_inputs(w, 1000 + idx, with_kv=False)
    gpu, wide = _accept_gpu_bf16(sv, _arrays(inp))
    compare_accept(gpu, wide, oracle.spec_accept(**wide))


def test_accept_streaming_vocabulary(sv):
    """A vocabulary above what one cluster holds on chip (262144) takes the
    streaming kernels with their statistics pre-pass."""
    V = 300000
    arrs = _synthetic_accept(31, 3, 7, V, [-1, 0, 0, 1, 1, 2, 2], sigma=2.0, noise=0.7)
    assert sv.spec_accept_workspace_size(3, 7, V) > 0
    gpu = _accept_gpu(sv, arrs)
    compare_accept(gpu, arrs, oracle.spec_accept(**arrs))


def test_accept_root_only_and_chain(sv):
    arrs = _synthetic_accept(21, 32, 1, 500, [-1])
    gpu = _accept_gpu(sv, arrs)
    orc = oracle.spec_accept(**arrs)
    compare_accept(gpu, arrs, orc)
    assert (gpu["accept_len"] == 0).all()
    # a lone root with several warps per CTA (V = 3001), clusters (40000,
    # 128256 with B = 24, the widest register slices) and the streamed walk
    # (300000): the root is a leaf, so every thread must see it as one
    for seed, B, V in ((24, 8, 3001), (25, 8, 40000), (27, 24, 128256), (26, 3, 300000)):
        arrs = _synthetic_accept(seed, B, 1, V, [-1])
        gpu = _accept_gpu(sv, arrs)
        compare_accept(gpu, arrs, oracle.spec_accept(**arrs))
        assert (gpu["accept_len"] == 0).all() and (gpu["status"] == 0).all()
        assert (gpu["out_tokens"][:, 0] >= 0).all()
    arrs = _synthetic_accept(22, 32, 12, 3000, chain_parent(12), sigma=1.0, noise=0.3)
    gpu = _accept_gpu(sv, arrs)
    compare_accept(gpu, arrs, oracle.spec_accept(**arrs))


@pytest.mark.parametrize("V,bf16", [(128256, False), (128255, False), (100000, True)])
def test_accept_wide_slices(sv, V, bf16):
    """Batches of 48 sequences at vocabularies where the widest 512-thread
    slices need more than one wave of clusters: for fp32 rows the library
    then takes the 352-thread, 16-slot slices when their smaller clusters
    need fewer waves (vector and scalar loads); bf16 rows keep the 512-thread
    slices at the same batch."""
    arrs = _synthetic_accept(60 + V % 11, 48, 7, V, [-1, 0, 0, 1, 1, 2, 2], sigma=2.0, noise=0.7)
    if bf16:
        gpu, wide = _accept_gpu_bf16(sv, arrs)
        compare_accept(gpu, wide, oracle.spec_accept(**wide))
    else:
        gpu = _accept_gpu(sv, arrs)
        compare_accept(gpu, arrs, oracle.spec_accept(**arrs))
    assert (gpu["status"] == 0).all()


@pytest.mark.parametrize("V", [3000, 40000])
def test_accept_star_tree(sv, V):
    """One node with 40 children and a second level below two of them: every
    child's token logits at the root's rows come from the threads that hold
    them, 40 pairs on one exchange; tokens drawn i.i.d. from q, so siblings
    repeat tokens."""
    parent = [-1] + [0] * 40 + [1] * 3 + [2] * 3
    arrs = _synthetic_accept(40 + V % 7, 16, len(parent), V, parent, sigma=1.0, noise=0.3)
    gpu = _accept_gpu(sv, arrs)
    compare_accept(gpu, arrs, oracle.spec_accept(**arrs))
    assert (gpu["status"] == 0).all()


def test_accept_status_errors(sv):
    arrs = _synthetic_accept(23, 4, 4, 100, [-1, 0, 0, 1])
    arrs["parent"][1, 2] = 3
    arrs["tokens"][2, 3] = 100
    arrs["tokens"][3, 1] = -5
    gpu = _accept_gpu(sv, arrs)
    orc = oracle.spec_accept(**arrs)
    assert gpu["status"].tolist() == orc["status"].tolist() == [0, 1, 2, 2]
    for b in (1, 2, 3):
        assert gpu["accept_len"][b] == 0
        assert (gpu["path"][b] == -1).all() and (gpu["out_tokens"][b] == -1).all()
        assert np.isnan(gpu["ratio"][b]).all()
    compare_accept(gpu, arrs, orc)


def test_accept_chi_square_on_gpu(sv):
    """One call with 10^6 sequences (V=8, chain of one draft drawn from q):
    the emitted token follows p (chi-square), and every trial matches the
    oracle bit for bit except near ties."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(31)
    V, B = 8, 1_000_000
    p = rng.dirichlet(np.ones(V)); q = rng.dirichlet(np.ones(V))
    lp, lq = np.log(p).astype(np.float32), np.log(q).astype(np.float32)
    qq = np.exp(lq.astype(np.float64) - lq.max()); qq /= qq.sum()
    pp = np.exp(lp.astype(np.float64) - lp.max()); pp /= pp.sum()
    tokens = np.zeros((B, 2), np.int32)
    tokens[:, 1] = rng.choice(V, size=B, p=qq)
    arrs = dict(target=np.broadcast_to(lp, (B, 2, V)).copy(),
                draft=np.broadcast_to(lq, (B, 2, V)).copy(), tokens=tokens,
                parent=np.broadcast_to(np.array([-1, 0], np.int32), (B, 2)).copy(),
                u_accept=rng.random((B, 2), dtype=np.float32),
                u_bonus=rng.random(B, dtype=np.float32))
    gpu = _accept_gpu(sv, arrs)
    counts = np.bincount(gpu["out_tokens"][:, 0], minlength=V)
    _, pval = chisquare(counts, pp * B)
    assert pval > 1e-4, pval
    orc = oracle.spec_accept(**arrs)
    compare_accept(gpu, arrs, orc, max_tie_frac=1e-3)


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------

def test_verify_step_tiny_chain(sv):
    w = WORKLOADS[0]
    inp = make_inputs(w, 1000)
    d = device_inputs(inp)
    out, lse, res, _ = sv.verify_step(d["parent"], d["tokens"], d["q"], d["k"], d["v"],
                                      d["page_table"], d["seq_lens"], d["target"], d["draft"],
                                      d["u_accept"], d["u_bonus"])
    torch.cuda.synchronize()
    o_ref, _ = oracle_attention(inp)
    assert np.abs(_np(out) - o_ref.reshape(out.shape)).max() <= F32_TOL
    arrs = _arrays(inp)
    compare_accept({k: (_np(v) if v is not None else None) for k, v in res.items()}, arrs,
                   oracle.spec_accept(**arrs))


# ---------------------------------------------------------------------------
# every chunk count (cluster size) on the same inputs
# ---------------------------------------------------------------------------

SPLIT_CASES = [
    # mixed lengths: short sequences leave some of a cluster's chunks empty
    ("bf16_mixed_lengths", 13, 10, "chain16",
     [40, 900, 120, 2000, 333, 64, 1500, 7, 250, 1100], 32, 8, 128, "bf16", 16),
    # one tile per sequence: every chunk but the first is empty
    ("single_node_no_prefix", 4, 2, "single", [0, 5], 4, 4, 128, "bf16", 128),
    # two row blocks of two halves, the tree inside the last tile
    ("random60_paged32_rowblocks", 3, 2, "random60", [700, 250], 8, 1, 128, "bf16", 32),
    ("binary31_g8_two_halves", 21, 3, "binary4", [3000, 65, 1200], 64, 8, 128, "bf16", 16),
]


@pytest.fixture
def force_splits(sv):
    lib = sv.load_library()
    yield lambda s: lib.svf_debug_set_attn_splits(s)
    lib.svf_debug_set_attn_splits(0)


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("case", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_attention_every_cluster_size(sv, force_splits, splits, case):
    name, seed, B, pk, lens, Hq, Hkv, D, dtype, ps = case
    assert force_splits(splits) == 0
    parent = _parent_of(pk, B, np.random.default_rng(seed + 100))
    N = parent.shape[1]
    c = _attn_case(seed, B, N, parent, lens, Hq, Hkv, D, dtype, ps)
    out, lse, status = _run_attn(sv, c, dtype)
    assert (status == 0).all()
    o_ref, l_ref = oracle.tree_attn(c["q"], c["K"], c["V"], c["lens"], c["parent"])
    err_o = np.abs(out - o_ref.reshape(out.shape)).max()
    err_l = np.abs(lse - l_ref.reshape(lse.shape)).max()
    print(f"{name} splits={splits}: max|out-ref| {err_o:.3g} max|lse-ref| {err_l:.3g}")
    assert err_o <= BF16_OUT_TOL and err_l <= BF16_LSE_TOL


@pytest.mark.parametrize("splits", [1, 2, 4, 8])
def test_attention_bad_inputs_every_cluster_size(sv, force_splits, splits):
    """A bad page id or a bad length zeroes that sequence's outputs (and sets
    its status) whatever the chunk count; the other sequences stay exact."""
    assert force_splits(splits) == 0
    B = 4
    parent = np.broadcast_to(binary_tree_parent(3), (B, 15)).copy()
    c = _attn_case(31, B, 15, parent, [900, 700, 1300, 400], 16, 4, 128, "bf16", 16)
    c["table"][1, 20] = c["P"] + 5          # a page id outside the cache
    lens = c["lens"].copy()
    lens[2] = 10 ** 6                        # longer than the page table
    c2 = dict(c, lens=lens)
    out, lse, status = _run_attn(sv, c2, "bf16")
    assert status.tolist() == [0, 4, 8, 0]
    for b in (1, 2):
        assert (out[b] == 0).all() and (lse[b] == 0).all()
    good = [0, 3]
    o_ref, _ = oracle.tree_attn(c["q"][good], c["K"][good], c["V"][good], c["lens"][good],
                                c["parent"][good])
    assert np.abs(out[good] - o_ref.reshape(out[good].shape)).max() <= BF16_OUT_TOL


# ---------------------------------------------------------------------------
# the persistent kernel: units split into pieces between CTAs
# ---------------------------------------------------------------------------

@pytest.fixture
def persistent(sv):
    lib = sv.load_library()
    assert lib.svf_debug_set_attn_kernel(2) == 0
    yield lib
    lib.svf_debug_set_attn_kernel(0)


def _check_attn(c, out, lse, status, skip=()):
    good = [b for b in range(c["q"].shape[0]) if b not in skip]
    assert (status[good] == 0).all(), status
    o_ref, l_ref = oracle.tree_attn(c["q"][good], c["K"][good], c["V"][good], c["lens"][good],
                                    c["parent"][good])
    err_o = np.abs(out[good] - o_ref.reshape(out[good].shape)).max()
    err_l = np.abs(lse[good] - l_ref.reshape(lse[good].shape)).max()
    assert err_o <= BF16_OUT_TOL and err_l <= BF16_LSE_TOL, (err_o, err_l)
    return err_o, err_l


PERSISTENT_CASES = [
    # one unit of 160 tiles: 20 CTAs of 8 tiles, every piece merged (F = 20)
    ("one_unit_twenty_pieces", 51, 1, "binary3", [10200], 4, 1, 128, 16),
    # four units of ~80 tiles over 40 CTAs: ~10 pieces per unit, both halves
    ("two_halves_ten_pieces", 52, 2, "binary4", [5000, 5100], 32, 2, 128, 16),
    # 300 short sequences (more than one CTA per SM): many whole units and
    # many segments per CTA, each with its own Q, tail tile and epilogue
    ("three_hundred_short", 53, 300, "chain16", None, 8, 2, 128, 16),
    # two row blocks of two halves (M = 480) and a contiguous cache
    ("row_blocks_contig", 54, 3, "random60", [3000, 90, 1500], 8, 1, 128, 0),
    # one tile per sequence: the tile space is shorter than the SM count
    ("tiny_units", 55, 5, "single", [0, 3, 10, 1, 40], 4, 4, 128, 16),
]


@pytest.mark.parametrize("case", PERSISTENT_CASES, ids=[c[0] for c in PERSISTENT_CASES])
def test_persistent_pieces_and_segments(sv, persistent, case):
    name, seed, B, pk, lens, Hq, Hkv, D, ps = case
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = rng.integers(0, 400, B).tolist()
    parent = _parent_of(pk, B, np.random.default_rng(seed + 100))
    c = _attn_case(seed, B, parent.shape[1], parent, lens, Hq, Hkv, D, "bf16", ps)
    out, lse, status = _run_attn(sv, c, "bf16", poison_tail=True)
    err_o, err_l = _check_attn(c, out, lse, status)
    print(f"{name}: max|out-ref| {err_o:.3g} max|lse-ref| {err_l:.3g}")


def test_persistent_bad_sequences_among_pieces(sv, persistent):
    """A bad page in the middle of a sequence whose units are split between
    CTAs zeroes every piece's merge of that sequence (the piece that saw the
    page flags it); a bad length has no tile at all. The rest stay exact."""
    B = 6
    parent = np.broadcast_to(binary_tree_parent(4), (B, 31)).copy()
    lens = [4000, 3000, 2500, 100, 3900, 700]
    c = _attn_case(61, B, 31, parent, lens, 64, 8, 128, "bf16", 16)
    c["table"][1, 100] = c["P"] + 3          # a page id outside the cache
    lens2 = c["lens"].copy()
    lens2[3] = 10 ** 6                        # longer than the page table
    c2 = dict(c, lens=lens2)
    out, lse, status = _run_attn(sv, c2, "bf16")
    assert status.tolist() == [0, 4, 0, 8, 0, 0], status
    for b in (1, 3):
        assert (out[b] == 0).all() and (lse[b] == 0).all()
    _check_attn(c, out, lse, status, skip=(1, 3))


def test_persistent_counters_reset_between_shapes(sv, persistent):
    """Calls of different shapes share one workspace: the per-unit counters
    each call leaves at zero must give the next call (another split of the
    tile space, other piece counts) exact results, and the first shape again
    after it."""
    ws_need = sv.tree_verify_attn_workspace_size(8, 31, 64, 8, 128, torch.bfloat16, 400, 16)
    ws = torch.zeros((ws_need,), dtype=torch.uint8, device="cuda")
    cases = []
    for seed, B, lens in ((71, 2, [6000, 2500]), (72, 8, [900, 50, 3000, 10, 2000, 700, 6300, 1]),
                          (71, 2, [6000, 2500])):
        parent = np.broadcast_to(binary_tree_parent(4), (B, 31)).copy()
        cases.append(_attn_case(seed, B, 31, parent, lens, 64, 8, 128, "bf16", 16))
    for c in cases:
        dev = "cuda"
        q = torch.from_numpy(c["q"]).to(dev).to(torch.bfloat16)
        kc = torch.from_numpy(c["kc"]).to(dev).to(torch.bfloat16)
        vc = torch.from_numpy(c["vc"]).to(dev).to(torch.bfloat16)
        anc, _, _ = sv.tree_mask_build(torch.from_numpy(c["parent"]).to(dev))
        for _ in range(2):
            out, lse, status = sv.tree_verify_attn(q, kc, vc, torch.from_numpy(c["table"]).to(dev),
                                                   torch.from_numpy(c["lens"]).to(dev), anc,
                                                   workspace=ws)
            torch.cuda.synchronize()
            _check_attn(c, _np(out.float()), _np(lse), _np(status))
    # every counter is back at zero: they are the workspace's last bytes
    units = 8 * 8
    assert (ws[ws_need - units * 8:].view(torch.int32) == 0).all()


def test_persistent_needs_a_workspace(sv, persistent):
    parent = np.broadcast_to(binary_tree_parent(2), (1, 7)).copy()
    c = _attn_case(81, 1, 7, parent, [100], 8, 2, 128, "bf16", 16)
    dev = "cuda"
    q = torch.from_numpy(c["q"]).to(dev).to(torch.bfloat16)
    kc = torch.from_numpy(c["kc"]).to(dev).to(torch.bfloat16)
    vc = torch.from_numpy(c["vc"]).to(dev).to(torch.bfloat16)
    anc, _, _ = sv.tree_mask_build(torch.from_numpy(c["parent"]).to(dev))
    with pytest.raises(sv.SpecVerifyError):
        sv.tree_verify_attn(q, kc, vc, torch.from_numpy(c["table"]).to(dev),
                            torch.from_numpy(c["lens"]).to(dev), anc,
                            workspace=torch.zeros((256,), dtype=torch.uint8, device=dev))


# ---------------------------------------------------------------------------
# the fused call: masks built inside the attention kernel
# ---------------------------------------------------------------------------

FUSED_CASES = [c for c in CASES if c[0] in ("worked_tree_contig", "binary31_paged16_g8",
                                            "random60_paged32_rowblocks", "single_node_no_prefix",
                                            "tree_crosses_tile", "fp32_d64", "bf16_mixed_lengths")]


@pytest.mark.parametrize("case", FUSED_CASES, ids=[c[0] for c in FUSED_CASES])
def test_fused_mask_attention_matches_the_two_calls(sv, attn_kernel, case):
    """svf_tree_mask_attn gives the masks of svf_tree_mask_build (checked
    against the oracle) and, bit for bit, the attention of
    svf_tree_verify_attn on those masks; one tree in the batch is invalid."""
    name, seed, B, pk, lens, Hq, Hkv, D, dtype, ps = case
    parent = _parent_of(pk, B, np.random.default_rng(seed + 100))
    N = parent.shape[1]
    if B > 1 and N > 1:
        parent[B - 1, N - 1] = N - 1          # not BFS: parent must precede the node
    c = _attn_case(seed, B, N, parent, lens, Hq, Hkv, D, dtype, ps)
    dev = "cuda"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.from_numpy(c["q"]).to(dev).to(tdt)
    kc = torch.from_numpy(c["kc"]).to(dev).to(tdt)
    vc = torch.from_numpy(c["vc"]).to(dev).to(tdt)
    table = torch.from_numpy(c["table"]).to(dev)
    sl = torch.from_numpy(c["lens"]).to(dev)
    par = torch.from_numpy(parent).to(dev)
    out_f, lse_f, st_f, anc_f, dep_f, mst_f = sv.tree_mask_attn(par, q, kc, vc, table, sl)
    anc, dep, mst = sv.tree_mask_build(par)
    out_s, lse_s, st_s = sv.tree_verify_attn(q, kc, vc, table, sl, anc)
    torch.cuda.synchronize()
    oa, od, os_ = oracle.tree_mask(parent)
    assert (_np(anc_f).view(np.uint64) == oa).all()
    assert (_np(dep_f) == od).all() and (_np(mst_f) == os_).all()
    assert torch.equal(st_f, st_s)
    assert torch.equal(out_f.view(torch.int16) if dtype == "bf16" else out_f,
                       out_s.view(torch.int16) if dtype == "bf16" else out_s)
    assert torch.equal(lse_f, lse_s)
