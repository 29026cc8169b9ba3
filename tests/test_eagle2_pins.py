"""Pins of the oracle's EAGLE-2 tree construction ("EAGLE 演化史", § E.2,
§ E.3 and the worked tree of § G; "The EAGLE Family", EAGLE-2).

Expected values come from the pages' worked tree (tests/golden/
worked_tree_7.json), from hand-computed products, and from invariants the
pages state: a node's value is the product of draft confidences on its root
path (recomputed here with scipy's softmax), and the top-N nodes by value
form a connected subtree.
"""

import json
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _rows_with(V, named, rest=None):
    """Logits whose softmax gives the named probabilities, the remaining mass
    spread evenly over the other tokens."""
    p = np.zeros(V)
    for t, q in named.items():
        p[t] = q
    others = [v for v in range(V) if v not in named]
    left = 1.0 - sum(named.values())
    for v in others:
        p[v] = left / len(others) if rest is None else rest
    with np.errstate(divide="ignore"):
        return np.maximum(np.log(p), -1e30).astype(np.float32)


def test_worked_tree_from_its_draft_rows(golden_dir):
    """§ G steps 1-3: the root's draft row gives 一 0.7, 五 0.2; 一's row gives
    百 0.6, 千 0.3; 五's row gives 百 0.4, 十 0.5. Two rounds with k = 2 and
    N = 7 keep everything; the flattened values are the page's products."""
    with open(os.path.join(golden_dir, "worked_tree_7.json")) as f:
        g = json.load(f)
    V = 8                       # 一 二 三 五 百 千 十 万 = 0..7
    YI, WU, BAI, QIAN, SHI = 0, 3, 4, 5, 6
    pool = oracle.eagle2_pool([7], 16)
    nxt, _ = oracle.eagle2_expand(pool, _rows_with(V, {YI: 0.7, WU: 0.2})[None, None],
                                  np.array([[0]]), 2)
    assert nxt.tolist() == [[1, 2]]
    rows = np.stack([_rows_with(V, {BAI: 0.6, QIAN: 0.3}), _rows_with(V, {BAI: 0.4, SHI: 0.5})])
    nxt, _ = oracle.eagle2_expand(pool, rows[None], nxt, 2)
    out = oracle.eagle2_finalize(pool, 7)
    assert out["n_out"][0] == 7 and out["connected"][0] == 1
    assert out["parent"][0].tolist() == g["parent"]
    # values by (parent token, token): the page lists 五's children as
    # [百 0.08, 十 0.10]; the rerank orders siblings by value, [十, 百]
    tok = out["token"][0]
    got = {(int(tok[out["parent"][0, i]]) if i else -1, int(tok[i])): out["value"][0, i]
           for i in range(7)}
    want = {(-1, 7): 1.0, (7, YI): 0.7, (7, WU): 0.2, (YI, BAI): 0.42, (YI, QIAN): 0.21,
            (WU, BAI): 0.08, (WU, SHI): 0.10}
    assert got.keys() == want.keys()
    for key, v in want.items():
        assert abs(got[key] - v) < 1e-6, key
    assert sorted(g["path_value"]) == pytest.approx(sorted(want.values()), abs=1e-6)


def test_expansion_step_weak_parent_strong_child():
    """§ E.3's phenomenon with feasible confidences: frontier values
    {0.95, 0.6, 0.3, 0.05}, k = 2. The two best are expanded; with top-2
    confidences {0.6, 0.3} and {0.5, 0.4} the children are worth
    {0.57, 0.285, 0.30, 0.24}, and the weaker parent's strong child (0.30)
    overtakes the stronger parent's weak child (0.285)."""
    V = 8
    pool = oracle.eagle2_pool([7], 32)
    # four children of the root, then their values set to the page's frontier
    nxt, _ = oracle.eagle2_expand(pool, _rows_with(V, {0: 0.4, 1: 0.3, 2: 0.2, 3: 0.1})[None, None],
                                  np.array([[0]]), 4)
    assert nxt.tolist() == [[1, 2, 3, 4]]
    pool["value"][0, 1:5] = [0.95, 0.6, 0.3, 0.05]
    rows = np.stack([_rows_with(V, {5: 0.6, 6: 0.3}), _rows_with(V, {6: 0.5, 7: 0.4})])
    nxt, gap = oracle.eagle2_expand(pool, rows[None], np.array([[1, 2]]), 2)
    np.testing.assert_allclose(pool["value"][0, 5:9], [0.57, 0.285, 0.30, 0.24], rtol=1e-6)
    assert nxt.tolist() == [[5, 7]]
    assert gap[0] == pytest.approx((0.30 - 0.285) / 0.30, rel=1e-5)


def _grow(rng, B, V, k, rounds, sigma=2.0):
    pool = oracle.eagle2_pool(rng.integers(0, V, size=B), 1 + k + (rounds - 1) * k * k)
    frontier = np.zeros((B, 1), np.int32)
    rows_of = {}
    for r in range(rounds):
        R = frontier.shape[1]
        rows = (sigma * rng.standard_normal((B, R, V))).astype(np.float32)
        for b in range(B):
            for i in range(R):
                if frontier[b, i] >= 0:
                    rows_of[(b, int(frontier[b, i]))] = rows[b, i]
        prev_count = pool["count"].copy()
        nxt, _ = oracle.eagle2_expand(pool, rows, frontier, k)
        # the next frontier is the top-k of this round's new nodes by value
        for b in range(B):
            new = np.arange(prev_count[b], pool["count"][b])
            vals = pool["value"][b, new]
            order = new[np.lexsort((new, -vals))][:k]
            assert nxt[b].tolist() == order.tolist()
        frontier = nxt
    return pool, rows_of


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_values_are_products_of_confidences_and_rerank_is_connected(seed):
    rng = np.random.default_rng(seed)
    B, V, k, rounds, N = 3, 50, 4, 4, 20
    pool, rows_of = _grow(rng, B, V, k, rounds)
    out = oracle.eagle2_finalize(pool, N)
    for b in range(B):
        n = out["n_out"][b]
        assert n == N and out["connected"][b] == 1
        par, tok, val, cid = (out[x][b] for x in ("parent", "token", "value", "cid"))
        # BFS order: parents first, depths non-decreasing, siblings by value
        depth = np.zeros(n, int)
        for i in range(1, n):
            assert 0 <= par[i] < i
            depth[i] = depth[par[i]] + 1
        assert (np.diff(depth) >= 0).all()
        for i in range(1, n - 1):
            if depth[i] == depth[i + 1]:
                assert par[i] <= par[i + 1]   # a level is grouped by parent, in order
            if par[i] == par[i + 1]:
                assert val[i] >= val[i + 1]
        # value = product of draft softmax probabilities along the root path
        for i in range(1, n):
            prob = softmax(rows_of[(b, int(cid[par[i]]))].astype(np.float64))
            assert val[i] == pytest.approx(val[par[i]] * prob[tok[i]], rel=1e-12)
            # the children of one node are its top-k draft tokens
            top = np.lexsort((np.arange(V), -prob))[:k]
            assert tok[i] in top
        # the kept nodes are the root and the N-1 best others by value
        allv = pool["value"][b, 1: pool["count"][b]]
        assert np.sort(val[1:])[::-1] == pytest.approx(np.sort(allv)[::-1][: N - 1], rel=1e-12)


def test_small_pool_and_gaps():
    """A pool smaller than N: every node is kept and the outputs are padded."""
    rng = np.random.default_rng(9)
    pool, _ = _grow(rng, 2, 20, 2, 2)
    out = oracle.eagle2_finalize(pool, 12)
    assert (out["n_out"] == 7).all()
    assert (out["parent"][:, 7:] == -1).all() and (out["token"][:, 7:] == -1).all()
    assert np.isinf(out["cut_gap"]).all()
