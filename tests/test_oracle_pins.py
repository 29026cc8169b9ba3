"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: every expected value is either
printed on the pages (the fixtures under tests/golden, each with its source),
a closed form, a brute-force enumeration, an independent library routine
(torch's scaled_dot_product_attention, networkx's ancestor sets, numpy's
searchsorted), or a distributional law checked by Monte Carlo / chi-square.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def anc_sets(anc_row):
    out = []
    for w, word in enumerate(anc_row):
        word = int(word)
        for bit in range(64):
            if word >> bit & 1:
                out.append(w * 64 + bit)
    return out


# ---------------------------------------------------------------------------
# O1: ancestor masks
# ---------------------------------------------------------------------------

def test_mask_worked_tree(golden_dir):
    g = load(golden_dir, "worked_tree_7.json")
    anc, depth, status = oracle.tree_mask(np.array(g["parent"]))
    assert status[0] == 0
    assert [anc_sets(anc[0, i]) for i in range(7)] == g["ancestors_or_self"]
    assert depth[0].tolist() == g["depth"]


def test_mask_brute_force_all_trees_up_to_7():
    nx = pytest.importorskip("networkx")
    for N in range(1, 8):
        for choice in itertools.product(*[range(i) for i in range(1, N)]):
            parent = np.array((-1,) + choice, dtype=np.int32)
            gph = nx.DiGraph()
            gph.add_nodes_from(range(N))
            gph.add_edges_from((int(parent[i]), i) for i in range(1, N))
            anc, depth, status = oracle.tree_mask(parent)
            assert status[0] == 0
            for i in range(N):
                expect = sorted(nx.ancestors(gph, i) | {i})
                assert anc_sets(anc[0, i]) == expect
                assert depth[0, i] == nx.shortest_path_length(gph, 0, i)


@pytest.mark.parametrize("d", [0, 1, 2, 3, 4, 5])
def test_mask_binary_tree_counts(d):
    from synth import binary_tree_parent
    parent = binary_tree_parent(d)
    assert parent.size == 2 ** (d + 1) - 1          # 31 nodes at depth 4
    anc, depth, status = oracle.tree_mask(parent)
    assert status[0] == 0
    for i in range(parent.size):
        assert len(anc_sets(anc[0, i])) == depth[0, i] + 1
        assert depth[0, i] == int(math.floor(math.log2(i + 1)))
    has_child = set(parent[1:].tolist())
    leaves = [i for i in range(parent.size) if i not in has_child]
    assert len(leaves) == 2 ** d


def test_mask_chain_is_causal():
    from synth import chain_parent
    for N in (1, 2, 16, 64, 100):
        anc, depth, status = oracle.tree_mask(chain_parent(N))
        for i in range(N):
            assert anc_sets(anc[0, i]) == list(range(i + 1))
            assert depth[0, i] == i


def test_mask_multiword_and_batch():
    rng = np.random.default_rng(1)
    N = 150
    parents = []
    for _ in range(3):
        p = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], dtype=np.int32)
        parents.append(p)
    parent = np.stack(parents)
    anc, depth, status = oracle.tree_mask(parent)
    assert anc.shape == (3, N, 3)
    for b in range(3):
        for i in (0, 1, 63, 64, 65, 149):
            chain = []
            a = i
            while a != -1:
                chain.append(a)
                a = parent[b, a]
            assert anc_sets(anc[b, i]) == sorted(chain)


def test_mask_invalid_parent_sets_status():
    bad = np.array([[0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, 0, 1]], dtype=np.int32)
    anc, depth, status = oracle.tree_mask(bad)
    assert status.tolist() == [1, 1, 1, 0]
    for b in range(3):
        for i in range(3):
            assert anc_sets(anc[b, i]) == [i] and depth[b, i] == 0


# ---------------------------------------------------------------------------
# O2: tree attention
# ---------------------------------------------------------------------------

def _random_attn_case(rng, B, N, Hq, Hkv, D, lens, parent):
    q = rng.standard_normal((B, N, Hq, D)).astype(np.float32)
    Tcap = int(max(lens)) + N
    k = rng.standard_normal((B, Tcap, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, Tcap, Hkv, D)).astype(np.float32)
    return q, k, v, np.array(lens, dtype=np.int32), parent


def _sdpa_causal(qs, ks, vs, scale):
    """Causal attention over one sequence with torch's library routine (fp64).

    qs [T, Hq, D], ks/vs [T, Hkv, D]; GQA by repeating KV heads.
    """
    Hq, Hkv = qs.shape[1], ks.shape[1]
    G = Hq // Hkv
    Q = torch.from_numpy(qs.astype(np.float64)).permute(1, 0, 2)[None]
    K = torch.from_numpy(ks.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    Vv = torch.from_numpy(vs.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()  # [T, Hq, D]


@pytest.mark.parametrize("case", ["worked", "random", "chain", "no_prefix"])
def test_attn_equals_causal_run_of_root_path(case):
    """Each node's output equals prompt + root->node path run as an ordinary
    causal sequence ("EAGLE 演化史" § B, correctness argument)."""
    rng = np.random.default_rng({"worked": 1, "random": 2, "chain": 3, "no_prefix": 4}[case])
    if case == "worked":
        parent = np.array([[-1, 0, 0, 1, 1, 2, 2]], dtype=np.int32)
        lens = [9]
    elif case == "random":
        N = 12
        parent = np.stack([np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)
                           for _ in range(2)])
        lens = [5, 17]
    elif case == "chain":
        parent = np.arange(-1, 5, dtype=np.int32)[None]
        lens = [7]
    else:
        parent = np.array([[-1, 0, 0, 1, 2, 2]], dtype=np.int32)
        lens = [0]
    B, N = parent.shape
    Hq, Hkv, D = 4, 2, 16
    q, k, v, lens, parent = _random_attn_case(rng, B, N, Hq, Hkv, D, lens, parent)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.tree_attn(q, k, v, lens, parent, scale)
    out = out.reshape(B, N, Hq, D)
    for b in range(B):
        L = int(lens[b])
        for i in range(N):
            path = []
            a = i
            while a != -1:
                path.append(a)
                a = parent[b, a]
            path = path[::-1]
            toks = list(range(L)) + [L + j for j in path]
            qs = np.concatenate([rng.standard_normal((L, Hq, D)).astype(np.float32),
                                 q[b, path]], axis=0)
            ref = _sdpa_causal(qs, k[b, toks], v[b, toks], scale)
            np.testing.assert_allclose(out[b, i], ref[-1], rtol=0, atol=1e-12)


def test_attn_chain_is_plain_causal_attention():
    rng = np.random.default_rng(5)
    N, L, Hq, Hkv, D = 6, 11, 8, 2, 32
    parent = np.arange(-1, N - 1, dtype=np.int32)[None]
    q, k, v, lens, parent = _random_attn_case(rng, 1, N, Hq, Hkv, D, [L], parent)
    out, _ = oracle.tree_attn(q, k, v, lens, parent)
    qs = np.concatenate([rng.standard_normal((L, Hq, D)).astype(np.float32), q[0]], 0)
    ref = _sdpa_causal(qs, k[0, : L + N], v[0, : L + N], 1 / math.sqrt(D))
    np.testing.assert_allclose(out.reshape(N, Hq, D), ref[L:], atol=1e-12, rtol=0)


def test_attn_single_node_is_decode_attention():
    rng = np.random.default_rng(6)
    L, Hq, Hkv, D = 40, 4, 4, 64
    q, k, v, lens, parent = _random_attn_case(rng, 1, 1, Hq, Hkv, D, [L],
                                              np.array([[-1]], np.int32))
    out, lse = oracle.tree_attn(q, k, v, lens, parent, 0.125)
    Q = torch.from_numpy(q[0].astype(np.float64)).permute(1, 0, 2)[None]     # [1,H,1,D]
    K = torch.from_numpy(k[0].astype(np.float64)).permute(1, 0, 2)[None]
    Vv = torch.from_numpy(v[0].astype(np.float64)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, scale=0.125)
    np.testing.assert_allclose(out, ref[0, :, 0].numpy(), atol=1e-12, rtol=0)
    s = (Q @ K.transpose(-1, -2))[0, :, 0] * 0.125
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)


def test_attn_equal_keys_closed_form():
    """With every key equal, all visible scores tie: the output is the mean of
    the visible values and lse = s + log(L + depth + 1)."""
    rng = np.random.default_rng(7)
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2, 3]], dtype=np.int32)
    N, L, Hq, Hkv, D = 8, 13, 2, 1, 8
    q, k, v, lens, parent = _random_attn_case(rng, 1, N, Hq, Hkv, D, [L], parent)
    kvec = rng.standard_normal(D).astype(np.float32)
    k[:] = kvec
    out, lse = oracle.tree_attn(q, k, v, lens, parent, 0.5)
    out = out.reshape(N, Hq, D)
    lse = lse.reshape(N, Hq)
    for i in range(N):
        vis = list(range(L))
        a = i
        depth = 0
        while a != -1:
            vis.append(L + a)
            a = parent[0, a]
            depth += 1
        for h in range(Hq):
            s = 0.5 * float(np.dot(q[0, i, h].astype(np.float64), kvec.astype(np.float64)))
            np.testing.assert_allclose(out[i, h], v[0, vis, 0].astype(np.float64).mean(0), atol=1e-12)
            assert abs(lse[i, h] - (s + math.log(L + depth))) < 1e-12


def test_attn_invalid_tree_sees_self_only():
    rng = np.random.default_rng(8)
    N, L, D = 4, 3, 8
    parent = np.array([[-1, 0, 5, 1]], dtype=np.int32)
    q, k, v, lens, parent = _random_attn_case(rng, 1, N, 1, 1, D, [L], parent)
    out, _ = oracle.tree_attn(q, k, v, lens, parent, 1.0)
    i = 3
    toks = list(range(L)) + [L + i]
    qs = np.concatenate([np.zeros((L, 1, D), np.float32), q[0, [i]]], 0)
    ref = _sdpa_causal(qs, k[0, toks], v[0, toks], 1.0)
    np.testing.assert_allclose(out[i], ref[-1, 0], atol=1e-12)


# ---------------------------------------------------------------------------
# O3: acceptance walk
# ---------------------------------------------------------------------------

def _row_from(named, V):
    p = np.zeros(V)
    for t, val in named.items():
        p[int(t)] = val
    rest = [t for t in range(V) if str(t) not in named]
    p[rest] = (1.0 - sum(named.values())) / len(rest)
    return np.log(p).astype(np.float32)


def _worked_inputs(g):
    V = len(g["vocab"])
    N = len(g["parent"])
    tgt = np.zeros((1, N, V), np.float32)
    dft = np.zeros((1, N, V), np.float32)
    for i in range(N):
        tgt[0, i] = _row_from(g["target_rows_named"].get(str(i), {}), V)
        dft[0, i] = _row_from(g["draft_rows_named"].get(str(i), {}), V)
    tokens = np.array([g["tree_tokens"]], np.int32)
    parent = np.array([g["parent"]], np.int32)
    ua = np.array([g["u_accept"]], np.float32)
    ub = np.array([g["u_bonus"]], np.float32)
    return tgt, dft, tokens, parent, ua, ub


def test_accept_worked_example(golden_dir):
    g = load(golden_dir, "accept_worked_example.json")
    r = oracle.spec_accept(*_worked_inputs(g))
    e = g["expected"]
    assert r["status"][0] == 0
    assert r["accept_len"][0] == e["accept_len"]
    assert r["path"][0, :3].tolist() == e["path"] and (r["path"][0, 3:] == -1).all()
    assert r["out_tokens"][0, :3].tolist() == e["out_tokens"] and (r["out_tokens"][0, 3:] == -1).all()
    assert abs(r["ratio"][0, 1] - e["ratio_node1"]) < 1e-6
    assert abs(r["ratio"][0, 3] - e["ratio_node3"]) < 1e-6
    assert abs(min(1.0, r["ratio"][0, 3]) - 0.917) < 5e-4      # the page's rounded figure
    # untested nodes carry NaN
    assert np.isnan(r["ratio"][0, [0, 2, 4, 5, 6]]).all()


def test_accept_worked_example_rejection_tries_sibling_with_residual(golden_dir):
    g = load(golden_dir, "accept_worked_example.json")
    tgt, dft, tokens, parent, ua, ub = _worked_inputs(g)
    ua[0, 3] = g["flip"]["u3"]
    r = oracle.spec_accept(tgt, dft, tokens, parent, ua, ub)
    f = g["flip"]
    assert r["path"][0, :3].tolist() == f["expected_path"]
    assert r["accept_len"][0] == f["expected_accept_len"]
    assert r["out_tokens"][0, :3].tolist() == f["expected_out_tokens"]
    assert abs(r["ratio"][0, 4] - f["expected_ratio_node4"]) < 1e-6


def _dist(rng, V, conc=1.0):
    return rng.dirichlet(np.full(V, conc))


def _logits(p):
    return np.log(p).astype(np.float32)


def _softmax64(l):
    e = np.exp(l.astype(np.float64) - l.max())
    return e / e.sum()


def _sample(rng, probs, n):
    return rng.choice(len(probs), size=n, p=probs).astype(np.int32)


def _chain_trials(rng, rows_p, rows_q, trials):
    """trials independent chains root->1->...->d; x_i ~ q_{i-1} i.i.d. per trial."""
    d = len(rows_p) - 1
    N = d + 1
    V = rows_p[0].size
    tgt = np.broadcast_to(np.stack([_logits(p) for p in rows_p]), (trials, N, V))
    dft = np.broadcast_to(np.stack([_logits(q) for q in rows_q]), (trials, N, V))
    tokens = np.zeros((trials, N), np.int32)
    qs = [_softmax64(_logits(q)) for q in rows_q]
    for i in range(1, N):
        tokens[:, i] = _sample(rng, qs[i - 1], trials)
    parent = np.broadcast_to(np.arange(-1, N - 1, dtype=np.int32), (trials, N))
    ua = rng.random((trials, N), dtype=np.float32)
    ub = rng.random(trials, dtype=np.float32)
    return oracle.spec_accept(tgt, dft, tokens, parent, ua, ub)


ALPHA_P = np.array([0.4, 0.3, 0.1, 0.1, 0.025, 0.025, 0.025, 0.025])
ALPHA_Q = np.array([0.1, 0.3, 0.3, 0.1, 0.05, 0.05, 0.05, 0.05])


@pytest.mark.parametrize("d", [4, 8])
def test_accept_chain_full_acceptance_is_alpha_pow_d(golden_dir, d):
    """Chain of depth d is fully accepted with probability prod_i sum_v min(p_i, q_i),
    alpha^d when every step overlaps by alpha ("EAGLE 演化史" § A: 0.24 at d=4,
    0.058 at d=8 for alpha=0.7)."""
    g = load(golden_dir, "acceptance_math.json")
    rng = np.random.default_rng(100 + d)
    p = _softmax64(_logits(ALPHA_P))
    q = _softmax64(_logits(ALPHA_Q))
    alpha = float(np.minimum(p, q).sum())
    assert abs(alpha - g["alpha"]) < 1e-6
    trials = 1_000_000
    r = _chain_trials(rng, [ALPHA_P] * (d + 1), [ALPHA_Q] * (d + 1), trials)
    full = float((r["accept_len"] == d).mean())
    expect = alpha ** d
    sigma = math.sqrt(expect * (1 - expect) / trials)
    assert abs(full - expect) < 4 * sigma
    page = g["chain_full_accept"][str(d)]
    assert abs(expect - page) < 0.5 * 10 ** -(len(str(page)) - 2)
    # expected accepted length: sum_{k=1..d} alpha^k
    el = sum(alpha ** kk for kk in range(1, d + 1))
    al = r["accept_len"].astype(np.float64)
    assert abs(al.mean() - el) < 4 * al.std() / math.sqrt(trials)


def test_accept_chain_distinct_rows_full_acceptance():
    rng = np.random.default_rng(11)
    V, d = 8, 3
    ps = [_dist(rng, V) for _ in range(d + 1)]
    qs = [_dist(rng, V) for _ in range(d + 1)]
    trials = 1_000_000
    r = _chain_trials(rng, ps, qs, trials)
    pp = [_softmax64(_logits(p)) for p in ps]
    qq = [_softmax64(_logits(q)) for q in qs]
    # P(accept_len >= k) = prod_{i<k} sum_v min(p_i, q_i)
    for kk in range(1, d + 1):
        expect = float(np.prod([np.minimum(pp[i], qq[i]).sum() for i in range(kk)]))
        got = float((r["accept_len"] >= kk).mean())
        assert abs(got - expect) < 4 * math.sqrt(expect * (1 - expect) / trials)


def _chisq_ok(samples, probs, min_p=1e-4):
    from scipy.stats import chisquare
    counts = np.bincount(samples, minlength=probs.size)
    _, pval = chisquare(counts, probs * counts.sum())
    return pval > min_p, pval


def test_accept_chi_square_first_token_is_target():
    """Lossless rule ("Eagle vs DFlash", speculative sampling): the emitted
    token is distributed as p whatever q is."""
    rng = np.random.default_rng(12)
    V = 8
    p, q = _dist(rng, V), _dist(rng, V)
    r = _chain_trials(rng, [p, _dist(rng, V)], [q, _dist(rng, V)], 1_000_000)
    ok, pval = _chisq_ok(r["out_tokens"][:, 0], _softmax64(_logits(p)))
    assert ok, pval


def test_accept_chi_square_second_token_given_first_accepted():
    rng = np.random.default_rng(13)
    V = 8
    ps = [_dist(rng, V) for _ in range(3)]
    qs = [_dist(rng, V) for _ in range(3)]
    r = _chain_trials(rng, ps, qs, 1_000_000)
    sel = r["accept_len"] >= 1
    ok, pval = _chisq_ok(r["out_tokens"][sel, 1], _softmax64(_logits(ps[1])))
    assert ok, pval


def _iid_sibling_trials(rng, p, q, k, trials, depth2=False):
    V = p.size
    if not depth2:
        N = 1 + k
        parent = np.array([-1] + [0] * k, np.int32)
    else:
        parent = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
        N = 7
    tgt = np.broadcast_to(_logits(p), (trials, N, V))
    dft = np.broadcast_to(_logits(q), (trials, N, V))
    qq = _softmax64(_logits(q))
    tokens = np.zeros((trials, N), np.int32)
    for c in range(1, N):
        tokens[:, c] = _sample(rng, qq, trials)
    ua = rng.random((trials, N), dtype=np.float32)
    ub = rng.random(trials, dtype=np.float32)
    return oracle.spec_accept(tgt, dft, tokens, np.broadcast_to(parent, (trials, N)), ua, ub)


def test_accept_chi_square_iid_siblings():
    """Multi-candidate rejection ("EAGLE 演化史" § C): with siblings drawn
    i.i.d. from the parent's draft softmax, the emitted token is still ~ p."""
    rng = np.random.default_rng(14)
    V = 8
    p, q = _dist(rng, V, 0.7), _dist(rng, V, 0.7)
    r = _iid_sibling_trials(rng, p, q, 3, 1_000_000)
    ok, pval = _chisq_ok(r["out_tokens"][:, 0], _softmax64(_logits(p)))
    assert ok, pval


def test_accept_binary_tree_level_probability_closed_form():
    """Two i.i.d. siblings per level: a level is passed with probability
    1 - (1-a1)(1-a2), a1 = sum min(p,q), a2 = sum min(r,q), r = max(0,p-q)/(1-a1)."""
    rng = np.random.default_rng(15)
    V = 8
    p, q = _dist(rng, V), _dist(rng, V)
    trials = 1_000_000
    r = _iid_sibling_trials(rng, p, q, 2, trials, depth2=True)
    pp, qq = _softmax64(_logits(p)), _softmax64(_logits(q))
    a1 = np.minimum(pp, qq).sum()
    res = np.maximum(pp - qq, 0) / (1 - a1)
    a2 = np.minimum(res, qq).sum()
    level = 1 - (1 - a1) * (1 - a2)
    for kk, expect in ((1, level), (2, level ** 2)):
        got = float((r["accept_len"] >= kk).mean())
        assert abs(got - expect) < 4 * math.sqrt(expect * (1 - expect) / trials)
    ok, pval = _chisq_ok(r["out_tokens"][:, 0], pp)
    assert ok, pval
    sel = r["accept_len"] >= 1
    ok, pval = _chisq_ok(r["out_tokens"][sel, 1], pp)
    assert ok, pval


def test_binary_bound_from_page(golden_dir):
    g = load(golden_dir, "acceptance_math.json")
    a, d = g["alpha"], 4
    bound = 1 - (1 - a ** d) ** (2 ** d)
    # the page prints the bound (0.98764) cut to two decimals
    assert math.floor(bound * 100) / 100 == g["binary_bound_d4"]
    assert 2 ** (d + 1) - 1 == g["binary_nodes"]["4"]


def test_accept_deterministic_candidate_is_not_lossless():
    """The rule is exact for i.i.d. candidates only: a candidate fixed to token 0
    with q=(1/2,1/2), p=(0.2,0.8) is emitted with probability min(1, .2/.5) = 0.4."""
    rng = np.random.default_rng(16)
    trials = 1_000_000
    p = np.array([0.2, 0.8]); q = np.array([0.5, 0.5])
    tgt = np.broadcast_to(_logits(p), (trials, 2, 2))
    dft = np.broadcast_to(_logits(q), (trials, 2, 2))
    tokens = np.zeros((trials, 2), np.int32)
    parent = np.broadcast_to(np.array([-1, 0], np.int32), (trials, 2))
    r = oracle.spec_accept(tgt, dft, tokens, parent, rng.random((trials, 2), dtype=np.float32),
                           rng.random(trials, dtype=np.float32))
    got = float((r["out_tokens"][:, 0] == 0).mean())
    assert abs(got - 0.4) < 4 * math.sqrt(0.24 / trials)
    # every rejection goes to token 1, the only token with residual mass
    assert (r["out_tokens"][r["accept_len"] == 0, 0] == 1).all()


def test_accept_root_only_is_inverse_cdf():
    rng = np.random.default_rng(17)
    V, trials = 50, 2000
    logits = (3 * rng.standard_normal((trials, 1, V))).astype(np.float32)
    u = rng.random(trials, dtype=np.float32)
    r = oracle.spec_accept(logits, logits, np.zeros((trials, 1), np.int32),
                           np.full((trials, 1), -1, np.int32), np.zeros((trials, 1), np.float32), u)
    assert (r["accept_len"] == 0).all() and (r["path"][:, 0] == 0).all()
    for t in range(trials):
        p = _softmax64(logits[t, 0])
        expect = int(np.searchsorted(np.cumsum(p), u[t] * p.sum(), side="right"))
        assert r["out_tokens"][t, 0] == expect


def test_accept_status_errors():
    V, N = 6, 3
    tgt = np.zeros((3, N, V), np.float32)
    dft = np.zeros((3, N, V), np.float32)
    tokens = np.array([[0, 1, 2], [0, 6, 2], [0, 1, -1]], np.int32)
    parent = np.array([[-1, 0, 0], [-1, 0, 2], [-1, 0, 1]], np.int32)
    r = oracle.spec_accept(tgt, dft, tokens, parent, np.full((3, N), .5, np.float32),
                           np.full(3, .5, np.float32))
    assert r["status"].tolist() == [0, 1 | 2, 2]
    for b in (1, 2):
        assert r["accept_len"][b] == 0
        assert (r["path"][b] == -1).all() and (r["out_tokens"][b] == -1).all()
    assert r["status"][0] == 0 and r["path"][0, 0] == 0


def test_accept_duplicate_sibling_after_rejection_is_rejected():
    """A sibling carrying the token its rejected twin carried has no residual
    mass on that token (p~ < q there before the subtraction)."""
    rng = np.random.default_rng(18)
    V = 8
    trials = 20000
    p, q = _dist(rng, V), _dist(rng, V)
    tgt = np.broadcast_to(_logits(p), (trials, 3, V))
    dft = np.broadcast_to(_logits(q), (trials, 3, V))
    x = _sample(rng, _softmax64(_logits(q)), trials)
    tokens = np.stack([np.zeros(trials, np.int32), x, x], 1)
    parent = np.broadcast_to(np.array([-1, 0, 0], np.int32), (trials, 3))
    r = oracle.spec_accept(tgt, dft, tokens, parent, rng.random((trials, 3), dtype=np.float32),
                           rng.random(trials, dtype=np.float32))
    assert not (r["path"][:, 1] == 2).any()
