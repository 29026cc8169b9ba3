"""Pins of the oracle's KV commit (rollback of rejected tree nodes).

"EAGLE-4 Technical Deepdive", § EAGLE-4 verification trees and harness, and
"EAGLE 演化史", § D.2: after verification the cache keeps the accepted
continuation and drops the rejected nodes' entries. The strongest pin is the
path-equivalence property of tree attention ("EAGLE 演化史", § B): once the
path is committed, running the committed sequence as an ordinary causal
sequence with torch's scaled_dot_product_attention must give, at every
committed position, the tree-attention output of the node that sits there.
That fixes which rows end up where, in which order, without reusing the
oracle's own copy logic.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle


def _paged(rng, B, lens, N, ps, Hkv, D, layers=1, spare=3, dtype=np.float32):
    """A paged cache with a random permuted page table; returns (k, v, table)."""
    need = [-(-(int(L) + N) // ps) for L in lens]
    max_pages = max(need) + 1
    num_pages = sum(need) + spare
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, np.int32)
    at = 0
    for b in range(B):
        table[b, : need[b]] = perm[at: at + need[b]]
        at += need[b]
    shape = (layers, num_pages, ps, Hkv, D)
    if dtype == np.uint16:
        k = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
        v = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    else:
        k = rng.standard_normal(shape).astype(np.float32)
        v = rng.standard_normal(shape).astype(np.float32)
    return k, v, table


def _logical(cache, table, b, T, ps):
    """Rows 0..T-1 of sequence b in token order (test-side page lookup)."""
    idx = np.arange(T)
    return cache[table[b, idx // ps], idx % ps]


def _random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)


def _root_path(parent, node):
    p = []
    while node != -1:
        p.append(int(node))
        node = parent[node]
    return p[::-1]


def _sdpa_causal(qs, ks, vs, scale):
    Hq, Hkv = qs.shape[1], ks.shape[1]
    G = Hq // Hkv
    Q = torch.from_numpy(qs.astype(np.float64)).permute(1, 0, 2)[None]
    K = torch.from_numpy(ks.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    Vv = torch.from_numpy(vs.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_commit_then_causal_attention_matches_tree_attention(seed):
    """After the commit, causal attention over the committed tokens at position
    L + k equals the tree-attention output of node path[k] computed on the
    cache before the commit, for every k."""
    rng = np.random.default_rng(100 + seed)
    B, N, Hq, Hkv, D, ps = 3, 13, 4, 2, 8, 4
    lens = np.array([5, 0, 11], np.int32)
    k, v, table = _paged(rng, B, lens, N, ps, Hkv, D)
    parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    q = rng.standard_normal((B, N, Hq, D)).astype(np.float32)
    path = np.full((B, N), -1, np.int32)
    alen = np.zeros(B, np.int32)
    for b in range(B):
        leaf = int(rng.integers(0, N))
        p = _root_path(parent[b], leaf)
        cut = int(rng.integers(1, len(p) + 1))  # any prefix of a root path is acceptable
        p = p[:cut]
        path[b, : len(p)] = p
        alen[b] = len(p) - 1
    # tree attention on the pre-commit cache, in logical order
    Tcap = int(lens.max()) + N
    kl = np.zeros((B, Tcap, Hkv, D), np.float32)
    vl = np.zeros((B, Tcap, Hkv, D), np.float32)
    for b in range(B):
        T = int(lens[b]) + N
        kl[b, :T] = _logical(k[0], table, b, T, ps)
        vl[b, :T] = _logical(v[0], table, b, T, ps)
    scale = 1.0 / math.sqrt(D)
    tree_out, _ = oracle.tree_attn(q, kl, vl, lens, parent, scale)
    tree_out = tree_out.reshape(B, N, Hq, D)

    res = oracle.kv_commit(k, v, table, lens, path, alen, N)
    assert (res["status"] == 0).all()
    np.testing.assert_array_equal(res["new_seq_lens"], lens + alen + 1)
    for b in range(B):
        L, n = int(lens[b]), int(alen[b]) + 1
        kc = _logical(res["k"][0], table, b, L + n, ps)
        vc = _logical(res["v"][0], table, b, L + n, ps)
        qs = np.concatenate([rng.standard_normal((L, Hq, D)).astype(np.float32),
                             q[b, path[b, :n]]], axis=0)
        ref = _sdpa_causal(qs, kc, vc, scale)
        for kk in range(n):
            np.testing.assert_allclose(ref[L + kk], tree_out[b, path[b, kk]], rtol=0, atol=1e-12)
        # the prefix is untouched, and so is everything past the committed tokens
        T = L + N
        before_k = _logical(k[0], table, b, T, ps)
        after_k = _logical(res["k"][0], table, b, T, ps)
        np.testing.assert_array_equal(after_k[:L], before_k[:L])
        np.testing.assert_array_equal(after_k[L + n:], before_k[L + n:])


def test_worked_walk_commit(golden_dir):
    """The page's worked walk accepts 一 then 百 (nodes 1 and 3 of the 7-node
    tree, "EAGLE 演化史" § G). Its committed sequence is prefix, root, node 1,
    node 3; nodes 2, 4, 5, 6 are rolled back."""
    with open(os.path.join(golden_dir, "accept_worked_example.json")) as f:
        g = json.load(f)
    path_nodes = g["expected"]["path"]
    N, L, ps, Hkv, D = len(g["parent"]), 3, 2, 1, 4
    # each token's row holds its own token index, so the layout can be read off
    num_pages = (L + N + ps - 1) // ps
    table = np.arange(num_pages, dtype=np.int32)[None]
    k = np.zeros((1, num_pages, ps, Hkv, D), np.float32)
    for t in range(L + N):
        k[0, t // ps, t % ps] = t
    v = -k
    path = np.full((1, N), -1, np.int32)
    path[0, : len(path_nodes)] = path_nodes
    res = oracle.kv_commit(k, v, table, np.array([L], np.int32), path,
                           np.array([g["expected"]["accept_len"]], np.int32), N)
    got = [int(res["k"][0, t // ps, t % ps, 0, 0]) for t in range(L + 3)]
    assert got == [0, 1, 2, L + 0, L + 1, L + 3]
    assert res["new_seq_lens"][0] == L + 3
    # tokens 0..5 fill pages 0-2; pages 3 and 4 held only rolled-back nodes
    assert res["n_freed"][0] == 2 and res["freed"][0].tolist()[:2] == [3, 4]
    np.testing.assert_array_equal(res["v"], -res["k"])


@pytest.mark.parametrize("alen", [0, 3, 6])
def test_chain_commit_moves_nothing(alen):
    """A chain's accepted path is 0..alen: every node is already in place."""
    rng = np.random.default_rng(7 + alen)
    N, ps = 7, 4
    lens = np.array([9], np.int32)
    k, v, table = _paged(rng, 1, lens, N, ps, 2, 8, layers=2)
    path = np.full((1, N), -1, np.int32)
    path[0, : alen + 1] = np.arange(alen + 1)
    res = oracle.kv_commit(k, v, table, lens, path, np.array([alen], np.int32), N)
    np.testing.assert_array_equal(res["k"], k)
    np.testing.assert_array_equal(res["v"], v)
    assert res["new_seq_lens"][0] == 9 + alen + 1


@pytest.mark.parametrize("L,N,ps,alen", [(0, 31, 16, 0), (5, 31, 16, 4), (15, 31, 16, 0),
                                         (16, 31, 16, 30), (1023, 16, 16, 15), (7, 5, 1, 2),
                                         (40, 60, 64, 3)])
def test_freed_pages_count_closed_form(L, N, ps, alen):
    """Pages past the committed tokens that held tree entries:
    ceil((L + N) / ps) - ceil((L + alen + 1) / ps), listed in table order."""
    rng = np.random.default_rng(L + N + ps)
    k, v, table = _paged(rng, 1, np.array([L]), N, ps, 1, 8)
    path = np.full((1, N), -1, np.int32)
    path[0, : alen + 1] = np.arange(alen + 1)
    res = oracle.kv_commit(k, v, table, np.array([L], np.int32), path,
                           np.array([alen], np.int32), N)
    first = -(-(L + alen + 1) // ps)
    end = -(-(L + N) // ps)
    assert res["n_freed"][0] == end - first
    assert res["freed"][0, : end - first].tolist() == table[0, first:end].tolist()
    assert (res["freed"][0, end - first:] == -1).all()
    assert end - first <= -(-N // ps)  # the row length the call needs


def test_layers_are_committed_alike():
    rng = np.random.default_rng(11)
    B, N, ps = 2, 9, 4
    lens = np.array([6, 2], np.int32)
    k, v, table = _paged(rng, B, lens, N, ps, 2, 8, layers=3)
    parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    path = np.full((B, N), -1, np.int32)
    alen = np.zeros(B, np.int32)
    for b in range(B):
        p = _root_path(parent[b], N - 1)
        path[b, : len(p)] = p
        alen[b] = len(p) - 1
    res = oracle.kv_commit(k, v, table, lens, path, alen, N)
    for layer in range(3):
        one = oracle.kv_commit(k[layer], v[layer], table, lens, path, alen, N)
        np.testing.assert_array_equal(res["k"][layer], one["k"])
        np.testing.assert_array_equal(res["v"][layer], one["v"])


def test_bf16_bit_patterns_move_unchanged():
    """2-byte elements (bf16 stored as uint16) are moved bit for bit."""
    rng = np.random.default_rng(12)
    N, ps = 8, 4
    lens = np.array([3], np.int32)
    k, v, table = _paged(rng, 1, lens, N, ps, 2, 8, dtype=np.uint16)
    path = np.full((1, N), -1, np.int32)
    path[0, :3] = [0, 2, 7]
    res = oracle.kv_commit(k, v, table, lens, path, np.array([2], np.int32), N)
    before = _logical(k[0], table, 0, 3 + N, ps)
    after = _logical(res["k"][0], table, 0, 3 + N, ps)
    np.testing.assert_array_equal(after[3:6], before[[3, 5, 10]])
    np.testing.assert_array_equal(after[6:], before[6:])


@pytest.mark.parametrize("case", ["len_high", "len_neg", "root", "order", "range", "length",
                                  "page"])
def test_bad_inputs_leave_the_cache_alone(case):
    rng = np.random.default_rng(13)
    N, ps = 6, 4
    lens = np.array([5], np.int32)
    k, v, table = _paged(rng, 1, lens, N, ps, 1, 8)
    path = np.array([[0, 1, 3, -1, -1, -1]], np.int32)
    alen = np.array([2], np.int32)
    expect = 32
    if case == "len_high":
        alen[0] = N
    elif case == "len_neg":
        alen[0] = -1
    elif case == "root":
        path[0, 0] = 1
    elif case == "order":
        path[0, 1:3] = [3, 1]
    elif case == "range":
        path[0, 2] = N
    elif case == "length":
        lens[0] = table.shape[1] * ps - N + 1
        expect = 8
    else:
        table[0, 1] = 10 ** 6
        expect = 4
    res = oracle.kv_commit(k, v, table, lens, path, alen, N)
    assert res["status"][0] == expect
    np.testing.assert_array_equal(res["k"], k)
    np.testing.assert_array_equal(res["v"], v)
    assert res["new_seq_lens"][0] == lens[0]
    assert res["n_freed"][0] == 0 and (res["freed"] == -1).all()
