"""GPU parity of the EAGLE-2 tree construction against the oracle, round by
round (pools and frontiers) and after the rerank (the flattened tree)."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

VALUE_RTOL = 2e-5   # fp32 softmax statistics against fp64, over up to 8 levels
NEAR_TIE = 1e-4     # relative gap below which two values may order either way


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


def _np(t):
    return t.detach().cpu().numpy()


def _build_both(sv, rng, B, V, k, rounds, N, capacity=None, sigma=2.0):
    """Grow the same tree on both sides from the same draft rows. Returns the
    GPU and oracle results and the sequences whose comparison stays exact (no
    near tie at any selection boundary)."""
    capacity = capacity or 1 + k + (rounds - 1) * k * k
    roots = rng.integers(0, V, size=B).astype(np.int32)
    gpool = sv.eagle2_pool(torch.from_numpy(roots).cuda(), capacity)
    opool = oracle.eagle2_pool(roots, capacity)
    frontier = np.zeros((B, 1), np.int32)
    exact = np.ones(B, bool)
    for _ in range(rounds):
        R = frontier.shape[1]
        rows = (sigma * rng.standard_normal((B, R, V))).astype(np.float32)
        status = torch.full((B,), -1, dtype=torch.int32).cuda()
        gnext = sv.eagle2_expand(gpool, torch.from_numpy(rows).cuda(),
                                 torch.from_numpy(frontier).cuda(), k, status=status)
        onext, gap = oracle.eagle2_expand(opool, rows, frontier, k)
        torch.cuda.synchronize()
        assert (_np(status) == 0).all()
        gn = _np(gnext)
        np.testing.assert_array_equal(_np(gpool["count"]), opool["count"])
        for b in range(B):
            if not exact[b]:
                continue
            c = opool["count"][b]
            for f in ("parent", "depth", "token"):
                np.testing.assert_array_equal(_np(gpool[f])[b, :c], opool[f][b, :c], err_msg=f)
            np.testing.assert_allclose(_np(gpool["value"])[b, :c], opool["value"][b, :c],
                                       rtol=VALUE_RTOL)
            if not (gn[b] == onext[b]).all():
                assert gap[b] < NEAR_TIE, f"sequence {b}: frontier {gn[b]} vs {onext[b]}"
                exact[b] = False
        frontier = onext  # both sides continue from the oracle's frontier
        if not exact.all():
            # the GPU pool diverged for those sequences: continue them from
            # the oracle's state so the remaining rounds still run
            for f in ("parent", "depth", "token", "value", "count"):
                gpool[f].copy_(torch.from_numpy(opool[f]).cuda())
    gout = sv.eagle2_finalize(gpool, N)
    oout = oracle.eagle2_finalize(opool, N)
    torch.cuda.synchronize()
    return gout, oout, exact


def _compare_final(gout, oout, exact):
    g = {k: _np(v) for k, v in gout.items()}
    np.testing.assert_array_equal(g["n_out"], oout["n_out"])
    flagged = 0
    for b in range(len(exact)):
        same = all((g[a][b] == oout[o][b]).all() for a, o in
                   (("parent", "parent"), ("tokens", "token"), ("cids", "cid")))
        if not same:
            assert oout["cut_gap"][b] < NEAR_TIE, f"sequence {b}: trees differ"
            flagged += 1
            continue
        np.testing.assert_allclose(g["values"][b], oout["value"][b], rtol=VALUE_RTOL)
    assert flagged <= max(1, len(exact) // 10)
    assert (oout["connected"] == 1).all()


@pytest.mark.parametrize("B,V,k,rounds,N", [
    (4, 128256, 8, 6, 60),      # the EAGLE-2 workload's shape
    (3, 32000, 4, 5, 31),
    (2, 1000, 1, 8, 9),         # k = 1: a chain
    (5, 5003, 16, 3, 100),
    (2, 16, 16, 2, 40),         # k = V
])
def test_eagle2_build_matches_oracle(sv, B, V, k, rounds, N):
    rng = np.random.default_rng(B * 1000 + k)
    gout, oout, exact = _build_both(sv, rng, B, V, k, rounds, N)
    _compare_final(gout, oout, exact)


def test_eagle2_small_capacity_and_padding(sv):
    """A pool too small for every child drops the rest; a tree smaller than
    N is padded."""
    rng = np.random.default_rng(3)
    gout, oout, exact = _build_both(sv, rng, 3, 300, 4, 3, 40, capacity=11)
    _compare_final(gout, oout, exact)
    assert (oout["n_out"] == 11).all()


def test_eagle2_worked_tree(sv):
    """The page's worked tree ("EAGLE 演化史", § G steps 1-3) built on the GPU."""
    V = 8
    def row(named):
        p = np.full(V, (1.0 - sum(named.values())) / (V - len(named)))
        for t, q in named.items():
            p[t] = q
        return np.log(p).astype(np.float32)
    pool = sv.eagle2_pool(torch.tensor([7], dtype=torch.int32).cuda(), 16)
    f = sv.eagle2_expand(pool, torch.from_numpy(row({0: 0.7, 3: 0.2})[None, None]).cuda(),
                         torch.zeros((1, 1), dtype=torch.int32).cuda(), 2)
    rows = np.stack([row({4: 0.6, 5: 0.3}), row({4: 0.4, 6: 0.5})])[None]
    sv.eagle2_expand(pool, torch.from_numpy(rows).cuda(), f, 2)
    out = sv.eagle2_finalize(pool, 7)
    torch.cuda.synchronize()
    assert _np(out["parent"])[0].tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert _np(out["tokens"])[0].tolist() == [7, 0, 3, 4, 5, 6, 4]
    np.testing.assert_allclose(_np(out["values"])[0], [1.0, 0.7, 0.2, 0.42, 0.21, 0.10, 0.08],
                               rtol=1e-6)


def _pattern_rows(rng, pattern, B, R, V):
    """Draft rows built to stress the top-k search: the candidate bound (every
    top value in one thread's elements), ties, and -inf logits."""
    rows = rng.standard_normal((B, R, V)).astype(np.float32)
    for b in range(B):
        for r in range(R):
            x = rows[b, r]
            if pattern == "constant":
                x[:] = 0.0
            elif pattern == "levels":       # a few values, many ties
                x[:] = rng.integers(0, 3, size=V)
            elif pattern == "descending":
                x[:] = np.linspace(4.0, -4.0, V, dtype=np.float32)
            elif pattern == "one_thread":
                # ids i0 + c + 4096 g (c, g < 4) share a thread in every
                # slicing of the row into multiples of 32 elements, and so do
                # the ids 16384 apart; give them the largest values
                i0 = 4 * int(rng.integers(0, 1000)) + 32064
                ids = [i0 + c + 4096 * g + 16384 * h for h in range(4) for g in range(4)
                       for c in range(4)]
                ids = [i for i in ids if i < V]
                x[ids] = 6.0 + rng.standard_normal(len(ids)).astype(np.float32)
            elif pattern == "few_finite":   # fewer finite logits than k
                keep = rng.choice(V, size=5, replace=False)
                y = np.full(V, -np.inf, np.float32)
                y[keep] = x[keep]
                x[:] = y
    return rows


@pytest.mark.parametrize("B,R", [(1, 1), (4, 8), (20, 8)])
@pytest.mark.parametrize("pattern", ["constant", "levels", "descending", "one_thread",
                                     "few_finite"])
def test_eagle2_expand_patterns(sv, B, R, pattern):
    """One expansion of R frontier rows per sequence; the rows per launch
    decide how many CTAs share a row (8, 4 and 1 for these shapes)."""
    V, k = 128256, 16
    rng = np.random.default_rng(sum(map(ord, pattern)) + B)
    cap = 1 + R + R * k
    roots = rng.integers(0, V, size=B).astype(np.int32)
    gpool = sv.eagle2_pool(torch.from_numpy(roots).cuda(), cap)
    opool = oracle.eagle2_pool(roots, cap)
    first = (2.0 * rng.standard_normal((B, 1, V))).astype(np.float32)
    frontier0 = np.zeros((B, 1), np.int32)
    sv.eagle2_expand(gpool, torch.from_numpy(first).cuda(), torch.from_numpy(frontier0).cuda(), R)
    front, _ = oracle.eagle2_expand(opool, first, frontier0, R)
    torch.cuda.synchronize()
    for f in ("parent", "depth", "token", "value", "count"):
        gpool[f].copy_(torch.from_numpy(opool[f]).cuda())   # start from the same pool
    rows = _pattern_rows(rng, pattern, B, R, V)
    gnext = sv.eagle2_expand(gpool, torch.from_numpy(rows).cuda(),
                             torch.from_numpy(front).cuda(), k)
    onext, gap = oracle.eagle2_expand(opool, rows, front, k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(gpool["count"]), opool["count"])
    for f in ("parent", "depth", "token"):
        np.testing.assert_array_equal(_np(gpool[f]), opool[f], err_msg=f)
    np.testing.assert_allclose(_np(gpool["value"]), opool["value"], rtol=VALUE_RTOL, atol=0)
    gn = _np(gnext)
    for b in range(B):
        if not (gn[b] == onext[b]).all():
            assert gap[b] < NEAR_TIE, f"sequence {b}: frontier {gn[b]} vs {onext[b]}"


@pytest.mark.parametrize("V,k", [(1 << 20, 16), (262147, 5)])
def test_eagle2_expand_large_vocab(sv, V, k):
    """The largest vocabulary (eight slices of eight batches per thread) and
    an odd one (element loads)."""
    rng = np.random.default_rng(V)
    gout, oout, exact = _build_both(sv, rng, 1, V, k, 2, 1 + k)
    _compare_final(gout, oout, exact)
