"""The acceptance comparison rules of gpu_common, checked on the CPU with
oracle results standing in for a GPU's: identical walks pass with no tie
taken, and planted differences far from any threshold fail."""

import numpy as np
import pytest

import oracle
from gpu_common import compare_accept, compare_onehot, decisions, residual_state, softmax64


def _case(seed, B=16, N=7, V=300):
    rng = np.random.default_rng(seed)
    tgt = (2.0 * rng.standard_normal((B, N, V))).astype(np.float32)
    dft = (tgt + 0.8 * rng.standard_normal((B, N, V))).astype(np.float32)
    parent = np.broadcast_to(np.array([-1, 0, 0, 1, 1, 2, 2], np.int32), (B, N)).copy()
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            tokens[b, c] = rng.choice(V, p=softmax64(dft[b, parent[b, c]]))
    return dict(target=tgt, draft=dft, tokens=tokens, parent=parent,
                u_accept=rng.random((B, N), dtype=np.float32),
                u_bonus=rng.random(B, dtype=np.float32))


def _as_gpu(orc):
    g = {k: np.array(orc[k]) for k in ("accept_len", "path", "out_tokens", "status")}
    g["ratio"] = orc["ratio"].astype(np.float32)
    return g


def test_identical_walks_pass_without_ties():
    a = _case(1)
    orc = oracle.spec_accept(**a)
    st = compare_accept(_as_gpu(orc), a, orc)
    assert st["walk_ties"] == 0 and st["bonus_ties"] == 0
    assert st["decisions"] > 0 and st["ratio_rel_err_first_tests"] < 1e-6


def test_a_far_bonus_token_fails():
    a = _case(2)
    orc = oracle.spec_accept(**a)
    g = _as_gpu(orc)
    b = int(np.argmax(orc["bonus_margin"]))
    g["out_tokens"][b, g["accept_len"][b]] = (g["out_tokens"][b, g["accept_len"][b]] + 1) % 300
    with pytest.raises(AssertionError):
        compare_accept(g, a, orc)


def test_a_far_decision_fails():
    a = _case(3)
    orc = oracle.spec_accept(**a)
    # a sequence whose first decision accepted with a clear margin
    for b in range(a["parent"].shape[0]):
        d = decisions(a["parent"][b], orc["ratio"][b], orc["path"][b], orc["accept_len"][b])
        if d and d[0][3] and orc["accept_margin"][b, d[0][0]] > 0.1:
            break
    else:
        pytest.skip("no clear first acceptance in this case")
    g = _as_gpu(orc)
    g["accept_len"][b] = 0
    g["path"][b, 1:] = -1
    g["out_tokens"][b, 1:] = -1
    g["ratio"][b, d[0][0] + 1:] = np.nan   # the GPU would have tested the next sibling
    with pytest.raises(AssertionError):
        compare_accept(g, a, orc)


def test_a_wrong_ratio_fails():
    a = _case(4)
    orc = oracle.spec_accept(**a)
    g = _as_gpu(orc)
    b, c = np.argwhere(~np.isnan(orc["ratio"]))[0]
    g["ratio"][b, c] *= 1.0 + 3e-5
    with pytest.raises(AssertionError):
        compare_accept(g, a, orc)


def test_residual_state_matches_the_literal_iteration():
    """The closed form used by the error model equals the pages' iteration
    p~ <- normalize(max(0, p~ - q)) after k rejections."""
    rng = np.random.default_rng(5)
    p, q = softmax64(rng.standard_normal(50)), softmax64(rng.standard_normal(50))
    pt = p.copy()
    for k in range(1, 4):
        r = np.maximum(0.0, pt - q)
        pt = r / r.sum()
        c, S = residual_state(p, q, k)
        np.testing.assert_allclose(np.maximum(0.0, p - c * q) / S, pt, rtol=1e-12, atol=1e-15)


def test_onehot_rules():
    a = _case(6)
    orc = oracle.spec_accept_onehot(a["target"], a["tokens"], a["parent"], a["u_accept"],
                                    a["u_bonus"])
    g = _as_gpu(dict(orc, n_rejects=None))
    assert compare_onehot(g, a["target"], a["tokens"], a["parent"], a["u_accept"], orc) == 0
    b, c = np.argwhere(~np.isnan(orc["ratio"]))[0]
    g["ratio"][b, c] *= 1.0 + 3e-5
    with pytest.raises(AssertionError):
        compare_onehot(g, a["target"], a["tokens"], a["parent"], a["u_accept"], orc)
