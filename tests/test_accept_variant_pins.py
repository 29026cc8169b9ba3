"""Pins of the oracle's target-only acceptance variants.

Greedy (temperature 0): "Eagle vs DFlash", § A fair evaluation protocol --
greedy speculative decoding must reproduce a target-only greedy run. Pinned
by that run itself (a chain whose drafts are the target's own argmaxes) and
by the temperature-0 limit of the stochastic rule, whose oracle is pinned in
test_oracle_pins.py.

One-hot candidates: the stochastic rule with q = one-hot(candidate). Pinned
by the stochastic oracle with one-hot draft rows on chains (where every
parent has one child, so both rules coincide), by a hand-worked case, and by
the property that makes it worth having: with deterministic (top-k)
siblings the emitted token is distributed as the target softmax (chi-square
over 10^6 trials), which the shared-q rule fails.
"""

import numpy as np
import pytest
from scipy.stats import chisquare

import oracle


def _random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)


def _greedy_case(rng, B, N, V, match=0.6):
    """Random trees whose children carry the parent's target argmax with
    probability `match` (otherwise another token), so paths get long."""
    tgt = (3.0 * rng.standard_normal((B, N, V))).astype(np.float32)
    parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            a = int(np.argmax(tgt[b, parent[b, c]]))
            tokens[b, c] = a if rng.random() < match else int((a + 1 + rng.integers(0, V - 1)) % V)
    return tgt, tokens, parent


def test_greedy_reproduces_a_target_only_run():
    """Drafts equal to the target's own greedy continuation are all accepted
    and the output is that continuation plus the next argmax; a draft that
    deviates at depth k stops the walk there."""
    rng = np.random.default_rng(1)
    N, V = 9, 50
    tgt = (2.0 * rng.standard_normal((1, N, V))).astype(np.float32)
    parent = np.arange(-1, N - 1, dtype=np.int32)[None]
    run = [int(np.argmax(tgt[0, i])) for i in range(N)]  # target-only greedy run
    tokens = np.array([[0] + run[: N - 1]], np.int32)
    r = oracle.spec_accept_greedy(tgt, tokens, parent)
    assert r["accept_len"][0] == N - 1
    assert r["out_tokens"][0].tolist() == run
    assert r["path"][0].tolist() == list(range(N))
    for k in range(1, N):
        bad = tokens.copy()
        bad[0, k] = (run[k - 1] + 1) % V
        r = oracle.spec_accept_greedy(tgt, bad, parent)
        assert r["accept_len"][0] == k - 1
        assert r["out_tokens"][0, :k].tolist() == run[:k]
        assert (r["out_tokens"][0, k:] == -1).all()


@pytest.mark.parametrize("seed", [2, 3])
def test_greedy_is_the_zero_temperature_limit_of_sampling(seed):
    """Logits scaled by 1e4 make every target softmax one-hot at its argmax;
    the stochastic rule then accepts a child iff it carries the argmax and
    draws the argmax as the bonus, whatever q and the uniforms are."""
    rng = np.random.default_rng(seed)
    B, N, V = 40, 15, 64
    tgt, tokens, parent = _greedy_case(rng, B, N, V)
    # no near-ties: the scaled argmax must be unique
    top2 = np.sort(tgt, axis=-1)[..., -2:]
    assert (top2[..., 1] - top2[..., 0] > 1e-4).all()
    g = oracle.spec_accept_greedy(tgt, tokens, parent)
    s = oracle.spec_accept(target=tgt * np.float32(1e4),
                           draft=(2.0 * rng.standard_normal((B, N, V))).astype(np.float32),
                           tokens=tokens, parent=parent,
                           u_accept=rng.random((B, N), dtype=np.float32),
                           u_bonus=rng.random(B, dtype=np.float32))
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(g[k], s[k], err_msg=k)
    assert g["accept_len"].max() >= 3


def test_greedy_duplicate_siblings_and_ties():
    """The first child (ascending index) carrying the argmax is taken; equal
    maxima resolve to the lowest token id."""
    V = 6
    tgt = np.zeros((1, 4, V), np.float32)
    tgt[0, 0] = [0, 5, 1, 5, 0, 0]     # tie between tokens 1 and 3: argmax 1
    tgt[0, 2] = [9, 0, 0, 0, 0, 0]
    tgt[0, 3] = [0, 0, 7, 0, 0, 0]
    parent = np.array([[-1, 0, 0, 0]], np.int32)
    tokens = np.array([[0, 3, 1, 1]], np.int32)    # node 1 carries 3, nodes 2 and 3 carry 1
    r = oracle.spec_accept_greedy(tgt, tokens, parent)
    assert r["path"][0].tolist() == [0, 2, -1, -1]
    assert r["out_tokens"][0].tolist() == [1, 0, -1, -1]


def test_greedy_invalid_inputs():
    tgt = np.zeros((2, 3, 5), np.float32)
    parent = np.array([[-1, 0, 0], [-1, 2, 0]], np.int32)
    tokens = np.array([[0, 1, 9], [0, 1, 1]], np.int32)
    r = oracle.spec_accept_greedy(tgt, tokens, parent)
    assert r["status"].tolist() == [2, 1]
    assert (r["path"] == -1).all() and (r["out_tokens"] == -1).all()
    assert (r["accept_len"] == 0).all()


def _one_hot_rows(tokens, parent, V):
    """Draft logits whose softmax at parent j is one-hot at its (only) child's
    token; rows of leaves are uniform and never read."""
    B, N = tokens.shape
    d = np.zeros((B, N, V), np.float32)
    for b in range(B):
        for c in range(1, N):
            j = parent[b, c]
            d[b, j] = -1e30
            d[b, j, tokens[b, c]] = 0.0
    return d


@pytest.mark.parametrize("seed", [4, 5])
def test_onehot_equals_sampling_with_one_hot_drafts_on_chains(seed):
    rng = np.random.default_rng(seed)
    B, N, V = 60, 8, 40
    tgt = (2.0 * rng.standard_normal((B, N, V))).astype(np.float32)
    parent = np.broadcast_to(np.arange(-1, N - 1, dtype=np.int32), (B, N)).copy()
    # children drawn from the target itself so that many are accepted
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            p = np.exp(tgt[b, c - 1].astype(np.float64))
            tokens[b, c] = rng.choice(V, p=p / p.sum())
    u = rng.random((B, N), dtype=np.float32)
    ub = rng.random(B, dtype=np.float32)
    h = oracle.spec_accept_onehot(tgt, tokens, parent, u, ub)
    s = oracle.spec_accept(target=tgt, draft=_one_hot_rows(tokens, parent, V), tokens=tokens,
                           parent=parent, u_accept=u, u_bonus=ub)
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(h[k], s[k], err_msg=k)
    tested = ~np.isnan(s["ratio"])
    np.testing.assert_allclose(h["ratio"][tested], s["ratio"][tested], rtol=1e-12)


def test_onehot_hand_case():
    """p = (0.5, 0.3, 0.2, 0) at the root, children carrying tokens 0 and 1,
    u = 0.6 and 0.5. Token 0: 0.6 < 0.5 fails, so p~ = (0, 0.6, 0.4, 0);
    token 1: 0.5 < 0.6 accepts. Node 2 is a leaf whose row puts all its mass
    on token 3, which is the bonus."""
    with np.errstate(divide="ignore"):
        tgt = np.log(np.array([[[0.5, 0.3, 0.2, 0.0], [0.25] * 4, [0.0, 0.0, 0.0, 1.0]]]))
    tgt = np.maximum(tgt, -1e30).astype(np.float32)
    parent = np.array([[-1, 0, 0]], np.int32)
    tokens = np.array([[0, 0, 1]], np.int32)
    r = oracle.spec_accept_onehot(tgt, tokens, parent, np.array([[0.0, 0.6, 0.5]], np.float32),
                                  np.array([0.3], np.float32))
    assert r["path"][0].tolist() == [0, 2, -1]
    assert r["out_tokens"][0].tolist() == [1, 3, -1]
    np.testing.assert_allclose(r["ratio"][0, 1:], [0.5, 0.6], rtol=1e-6)


def test_onehot_is_lossless_for_deterministic_siblings():
    """Depth-1 tree, three children fixed to the draft's top-3 tokens (no
    sampling): the emitted token must follow the target softmax p_0."""
    rng = np.random.default_rng(6)
    V, T = 8, 1_000_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    top3 = np.argsort(-q)[:3].astype(np.int32)
    tgt = np.broadcast_to(np.log(p).astype(np.float32), (T, 4, V))
    parent = np.broadcast_to(np.array([-1, 0, 0, 0], np.int32), (T, 4))
    tokens = np.broadcast_to(np.concatenate([[0], top3]).astype(np.int32), (T, 4))
    u = rng.random((T, 4), dtype=np.float32)
    ub = rng.random(T, dtype=np.float32)
    r = oracle.spec_accept_onehot(tgt, tokens, parent, u, ub)
    counts = np.bincount(r["out_tokens"][:, 0], minlength=V)
    _, pval = chisquare(counts, p * T)
    assert pval > 1e-4, pval
