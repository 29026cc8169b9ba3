"""Input generator: tree builders pinned on the pages' worked examples, and
structural invariants of every workload (no verification arithmetic here)."""

import json
import os

import numpy as np
import pytest

from synth import (WORKLOADS, binary_tree_parent, build_eagle2_tree, chain_parent,
                   eagle2_expand_step, f32_to_bf16_bits, bf16_bits_to_f32, make_tree)
from synth.gen import draft_probs, page_layout, prefix_lengths, logical_kv, make_inputs


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_eagle2_expand_step_worked_example(golden_dir):
    g = load(golden_dir, "eagle2_step.json")
    sel, children, frontier = eagle2_expand_step(g["frontier_values"], g["child_confidences"], g["k"])
    assert sel.tolist() == g["expected_expanded_positions"]
    np.testing.assert_allclose(children, g["expected_children_values"], atol=1e-12)
    np.testing.assert_allclose(frontier, g["expected_new_frontier"], atol=1e-12)


def _rows_from_conf(conf_by_cid, V):
    """Draft logits whose softmax puts the given confidences on given tokens."""
    def row_of(cid):
        named = conf_by_cid.get(cid, {})
        p = np.full(V, (1.0 - sum(named.values())) / (V - len(named)))
        for t, c in named.items():
            p[t] = c
        return np.log(p)
    return row_of


def test_eagle2_builder_reproduces_worked_tree(golden_dir):
    """Two expansion rounds of width 2 give the page's 7-node tree with path
    values [1.0, 0.7, 0.2, 0.42, 0.21, 0.08, 0.10] ("EAGLE 演化史" § G)."""
    g = load(golden_dir, "worked_tree_7.json")
    V = 64
    # token ids: 一=1, 五=5, 百=10, 千=11, 十=12; creation ids: root 0, 一 1, 五 2
    conf = {0: {1: 0.7, 5: 0.2}, 1: {10: 0.6, 11: 0.3}, 2: {10: 0.4, 12: 0.5}}
    parent, cids, tokens, values = build_eagle2_tree(_rows_from_conf(conf, V), 0, topk=2,
                                                     rounds=2, n_nodes=7)
    name = {0: "root", 1: "一", 5: "五", 10: "百", 11: "千", 12: "十"}
    got = {}
    for i in range(7):
        key = (name[int(tokens[parent[i]])] if parent[i] >= 0 else None, name[int(tokens[i])])
        got[key] = values[i]
    want = {}
    for i in range(7):
        pi = g["parent"][i]
        key = (g["tokens"][pi] if pi >= 0 else None, g["tokens"][i])
        want[key] = g["path_value"][i]
    assert got.keys() == want.keys()
    for k in want:
        assert abs(got[k] - want[k]) < 1e-9
    # BFS order: parents precede children; siblings in descending draft confidence
    assert parent.tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert [name[int(t)] for t in tokens] == ["root", "一", "五", "百", "千", "十", "百"]


def test_eagle2_top_n_is_connected_subtree():
    rng = np.random.default_rng(3)
    V = 40
    for trial in range(20):
        rows = {}

        def row_of(cid):
            if cid not in rows:
                rows[cid] = 2.0 * rng.standard_normal(V)
            return rows[cid]

        parent, cids, tokens, values = build_eagle2_tree(row_of, 0, topk=4, rounds=4, n_nodes=25)
        assert parent[0] == -1
        for i in range(1, 25):
            assert 0 <= parent[i] < i
            assert values[parent[i]] >= values[i]


def test_chain_and_binary_parents():
    assert chain_parent(4).tolist() == [-1, 0, 1, 2]
    assert binary_tree_parent(2).tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert binary_tree_parent(4).size == 31


def test_bf16_round_trip_and_rne():
    x = np.array([1.0, -2.5, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 3.14159], np.float32)
    b = f32_to_bf16_bits(x)
    y = bf16_bits_to_f32(b)
    assert y[0] == 1.0 and y[1] == -2.5
    assert y[2] == 1.0                       # halfway, rounds to even
    assert y[3] == 1.0 + 2 ** -7             # above halfway rounds up
    assert abs(y[4] - 3.140625) < 1e-7


@pytest.mark.parametrize("idx", [0, 1, 3])
def test_workload_tree_and_layout_invariants(idx):
    w = WORKLOADS[idx]
    seed = 1000 + idx
    inp = make_inputs(w, seed, with_kv=(idx < 2), with_logits=(idx < 2))
    assert inp.parent.shape == (w.B, w.N)
    for b in range(w.B):
        p = inp.parent[b]
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, w.N))
    if w.tree == "binary":
        # children of j are the top-2 draft tokens of j, highest first
        for j in range(3):
            q = draft_probs(inp.draft[0, j]) if inp.draft is not None else None
            if q is not None:
                top = np.lexsort((np.arange(q.size), -q))[:2]
                assert inp.tokens[0, 2 * j + 1] == top[0] and inp.tokens[0, 2 * j + 2] == top[1]
    # every logical token maps to a distinct (page, slot)
    T = inp.seq_lens.astype(np.int64) + w.N
    seen = set()
    for b in range(w.B):
        for t in range(int(T[b])):
            page = int(inp.page_table[b, t // inp.page_size])
            assert 0 <= page < inp.num_pages
            key = (page, t % inp.page_size)
            assert key not in seen
            seen.add(key)
    assert ((inp.u_accept >= 0) & (inp.u_accept < 1)).all()


def test_paged_cache_holds_logical_values():
    w = WORKLOADS[3]
    seed = 1003
    inp = make_inputs(w, seed, with_kv=True, with_logits=False, workers=1)
    for b, g in ((0, 0), (5, 7)):
        T = int(inp.seq_lens[b]) + w.N
        k, v = logical_kv(w, seed, b, g, T)
        t = np.arange(T)
        pages = inp.page_table[b, t // inp.page_size]
        np.testing.assert_array_equal(inp.k_cache[pages, t % inp.page_size, g], k)
        np.testing.assert_array_equal(inp.v_cache[pages, t % inp.page_size, g], v)


def test_eagle2_workload_shape():
    w = WORKLOADS[2]
    parent, keys, tokens = make_tree(w, 1002, 0)
    assert parent.size == 60
    depth = np.zeros(60, int)
    for i in range(1, 60):
        depth[i] = depth[parent[i]] + 1
    assert depth.max() <= 6
    assert (np.diff(depth) >= 0).all()       # BFS order
