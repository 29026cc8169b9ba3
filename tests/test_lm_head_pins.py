"""Pins of the oracle's LM head and of the acceptance walk fed by it (the
fused LM head + acceptance row), each against something other than the
oracle's own formula: exact special cases, closed forms and the page's
worked walk."""

import numpy as np
import pytest

import oracle
from test_oracle_pins import _worked_inputs, load


def test_one_hot_weight_rows_select_hidden_components():
    """Row v of W = e_pi(v): logit v of node r is h[r][pi(v)], bit for bit."""
    rng = np.random.default_rng(0)
    R, H, V = 5, 16, 40
    h = rng.standard_normal((R, H)).astype(np.float32)
    pi = rng.integers(0, H, size=V)
    W = np.zeros((V, H), np.float32)
    W[np.arange(V), pi] = 1.0
    out = oracle.lm_head_logits(h, W)
    np.testing.assert_array_equal(out, h[:, pi].astype(np.float64))


def test_constant_rows_closed_form():
    """h[r] = a_r for every component, W[v] = c_v: logit = H a_r c_v."""
    H = 4096
    a = np.array([1, -2, 3], np.float32)
    c = np.array([0.5, -0.25, 2, 0, 7], np.float32)
    h = np.repeat(a[:, None], H, axis=1)
    W = np.repeat(c[:, None], H, axis=1)
    out = oracle.lm_head_logits(h[None], W)[0]
    np.testing.assert_array_equal(out, H * np.outer(a, c).astype(np.float64))


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((3, 7, 64)).astype(np.float32)
    W = rng.standard_normal((100, 64)).astype(np.float32)
    np.testing.assert_array_equal(oracle.lm_head_logits(h, 2 * W),
                                  2 * oracle.lm_head_logits(h, W))


def test_orthonormal_head_gives_the_identity():
    """W = Q with orthonormal rows (numpy's QR builds it) and h = Q's rows:
    the logits are the identity matrix."""
    rng = np.random.default_rng(2)
    H = 48
    Q, _ = np.linalg.qr(rng.standard_normal((H, H)))
    Qf = Q.T.astype(np.float32)          # rows orthonormal (to float32 rounding)
    out = oracle.lm_head_logits(Qf, Qf)
    np.testing.assert_allclose(out, np.eye(H), atol=2e-6)


def test_transposed_roles():
    """logits(h, W) = logits(W, h) transposed: every product is the same dot."""
    rng = np.random.default_rng(3)
    h = rng.standard_normal((6, 32)).astype(np.float32)
    W = rng.standard_normal((9, 32)).astype(np.float32)
    np.testing.assert_array_equal(oracle.lm_head_logits(h, W), oracle.lm_head_logits(W, h).T)


def test_identity_head_reduces_to_the_walk(golden_dir):
    """With V = H and W = I the LM head returns the hidden states, so the
    fused walk on the page's worked tree must give the page's result (path
    root -> 1 -> 3, three tokens, ratios 1 and 0.917)."""
    g = load(golden_dir, "accept_worked_example.json")
    tgt, dft, tokens, parent, ua, ub = _worked_inputs(g)
    V = tgt.shape[-1]
    r = oracle.spec_accept_lmhead(tgt, np.eye(V, dtype=np.float32), dft, tokens, parent, ua, ub)
    np.testing.assert_array_equal(r["target"], tgt)
    e = g["expected"]
    assert r["accept_len"][0] == e["accept_len"]
    assert r["path"][0, :3].tolist() == e["path"]
    assert r["out_tokens"][0, :3].tolist() == e["out_tokens"]
    assert abs(min(1.0, r["ratio"][0, 3]) - 0.917) < 5e-4


@pytest.mark.parametrize("seed", [4, 5])
def test_permuted_head_permutes_the_emitted_tokens(seed):
    """Relabelling the vocabulary (W's rows permuted) relabels every token:
    with the draft rows and tree tokens permuted alike, the fused walk takes
    the same path and emits the relabelled tokens. Uniforms are shared."""
    rng = np.random.default_rng(seed)
    B, N, H, V = 4, 7, 24, 24
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2]] * B, np.int32)
    hidden = (2 * rng.standard_normal((B, N, H))).astype(np.float32)
    W = np.eye(V, dtype=np.float32)
    draft = (oracle.lm_head_logits(hidden, W) + rng.standard_normal((B, N, V))).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    ua = rng.random((B, N), dtype=np.float32)
    ub = rng.random(B, dtype=np.float32)
    base = oracle.spec_accept_lmhead(hidden, W, draft, tokens, parent, ua, ub)
    perm = rng.permutation(V)            # token v becomes perm[v]
    inv = np.argsort(perm)
    Wp = W[inv]                          # new row perm[v] holds old row v
    r = oracle.spec_accept_lmhead(hidden, Wp, draft[..., inv], perm[tokens].astype(np.int32),
                                  parent, ua, ub)
    np.testing.assert_array_equal(r["path"], base["path"])
    np.testing.assert_array_equal(r["accept_len"], base["accept_len"])
    # accepted draft tokens relabel exactly; the bonus token is drawn by an
    # inverse CDF over the relabelled order, so only its validity is checked
    for b in range(B):
        n = base["accept_len"][b]
        assert r["out_tokens"][b, :n].tolist() == perm[base["out_tokens"][b, :n]].tolist()
        assert 0 <= r["out_tokens"][b, n] < V
