"""GPU parity of the target-only acceptance variants (greedy, one-hot
candidates) against the oracle."""

import math

import numpy as np
import pytest
import torch
from scipy.stats import chisquare

import oracle
from gpu_common import compare_onehot

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


def _np(t):
    return None if t is None else t.detach().cpu().numpy()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)


def _case(seed, B, N, V, topk_children=True, sigma=3.0, noise=1.0, binary=False):
    """Target rows ~ N(0, sigma^2); children carry the top tokens of a draft row
    (target + noise) at their parent, in sibling order, so greedy and one-hot
    walks go deep."""
    rng = np.random.default_rng(seed)
    tgt = (sigma * rng.standard_normal((B, N, V))).astype(np.float32)
    if binary:
        parent = np.broadcast_to(np.array([-1] + [(i - 1) // 2 for i in range(1, N)], np.int32),
                                 (B, N)).copy()
    else:
        parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for j in range(N):
            kids = np.nonzero(parent[b] == j)[0]
            if len(kids) == 0:
                continue
            d = tgt[b, j] + noise * rng.standard_normal(V).astype(np.float32)
            if topk_children:
                order = np.argsort(-d, kind="stable")[: len(kids)]
            else:
                order = rng.integers(0, V, size=len(kids))
            tokens[b, kids] = order
    return dict(target=tgt, tokens=tokens, parent=parent,
                u_accept=rng.random((B, N), dtype=np.float32),
                u_bonus=rng.random(B, dtype=np.float32))


def _greedy(sv, a):
    r = sv.spec_accept_greedy(_dev(a["target"]), _dev(a["tokens"]), _dev(a["parent"]))
    torch.cuda.synchronize()
    return {k: _np(v) for k, v in r.items()}


def _onehot(sv, a):
    r = sv.spec_accept_onehot(_dev(a["target"]), _dev(a["tokens"]), _dev(a["parent"]),
                              _dev(a["u_accept"]), _dev(a["u_bonus"]))
    torch.cuda.synchronize()
    return {k: _np(v) for k, v in r.items()}


def _compare_onehot(gpu, orc, a):
    """Bit-exact except near ties under the one-hot error model (gpu_common)."""
    return compare_onehot(gpu, a["target"], a["tokens"], a["parent"], a["u_accept"], orc)


VOCABS = [8, 37, 1000, 4096, 5003, 32000, 128256, 151936]


@pytest.mark.parametrize("V", VOCABS)
def test_greedy_matches_oracle(sv, V):
    B = 24 if V > 100000 else 64
    a = _case(V, B, 15, V, noise=0.5)
    gpu = _greedy(sv, a)
    orc = oracle.spec_accept_greedy(a["target"], a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(gpu[k], orc[k], err_msg=k)
    assert orc["accept_len"].max() >= 2


@pytest.mark.parametrize("V", VOCABS)
def test_onehot_matches_oracle(sv, V):
    B = 24 if V > 100000 else 64
    # a flat softmax over a large vocabulary accepts nothing: peak it there
    a = _case(V + 7, B, 15, V, sigma=2.0 if V <= 5003 else 8.0, noise=0.7)
    gpu = _onehot(sv, a)
    orc = oracle.spec_accept_onehot(a["target"], a["tokens"], a["parent"], a["u_accept"],
                                    a["u_bonus"])
    _compare_onehot(gpu, orc, a)
    assert orc["accept_len"].max() >= 1


# above 262144 the rows stream from memory (accept_target_stream.cu); 262145
# and 300001 take the scalar loads (V % 4 != 0), 786432 is the largest
STREAM_VOCABS = [262145, 300000, 300001, 524288, 786432]


@pytest.mark.parametrize("V", STREAM_VOCABS)
def test_greedy_streaming_vocabularies(sv, V):
    # the top gaps of 3e5 draws are small: little draft noise, so walks go deep
    a = _case(V, 6, 15, V, noise=0.05)
    gpu = _greedy(sv, a)
    orc = oracle.spec_accept_greedy(a["target"], a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(gpu[k], orc[k], err_msg=k)
    assert orc["accept_len"].max() >= 2


@pytest.mark.parametrize("V", STREAM_VOCABS)
def test_onehot_streaming_vocabularies(sv, V):
    a = _case(V + 7, 4, 15, V, sigma=8.0, noise=0.7)
    gpu = _onehot(sv, a)
    orc = oracle.spec_accept_onehot(a["target"], a["tokens"], a["parent"], a["u_accept"],
                                    a["u_bonus"])
    _compare_onehot(gpu, orc, a)
    assert orc["accept_len"].max() >= 1


def test_onehot_streaming_flat_rows_bonus(sv):
    """Flat rows over 524288 tokens: every child is rejected, so every
    sequence's bonus token comes from the inverse CDF of the residual over the
    whole streamed row, with the rejected tokens excluded."""
    a = _case(77, 6, 7, 524288, sigma=1.0, noise=0.7)
    gpu = _onehot(sv, a)
    orc = oracle.spec_accept_onehot(a["target"], a["tokens"], a["parent"], a["u_accept"],
                                    a["u_bonus"])
    _compare_onehot(gpu, orc, a)


def test_variants_streaming_status_and_duplicates(sv):
    V = 300000
    a = _case(55, 4, 7, V)
    a["tokens"][1, 4] = V          # outside the vocabulary
    a["parent"][2] = [-1, 0, 1, 2, 3, 4, 5]   # a chain
    a["tokens"][2, 1:] = 7         # duplicate tokens along it
    a["parent"][3] = [-1, 0, 0, 0, 0, 0, 0]   # five siblings, two with the same token
    a["tokens"][3, 2] = a["tokens"][3, 1]
    for run, ref in ((_greedy, lambda: oracle.spec_accept_greedy(a["target"], a["tokens"],
                                                                  a["parent"])),
                     (_onehot, lambda: oracle.spec_accept_onehot(**a))):
        gpu = run(sv, a)
        orc = ref()
        assert gpu["status"].tolist() == orc["status"].tolist() == [0, 2, 0, 0]
        assert (gpu["path"][1] == -1).all() and gpu["accept_len"][1] == 0
        if run is _greedy:
            for k in ("accept_len", "path", "out_tokens"):
                np.testing.assert_array_equal(gpu[k], orc[k], err_msg=k)
        else:
            _compare_onehot(gpu, orc, a)


def test_variants_many_sequences(sv):
    """More sequences than SMs at the 70B-serving vocabulary: binary trees."""
    a = _case(99, 64, 31, 128256, noise=1.5, binary=True)
    g = _greedy(sv, a)
    o = oracle.spec_accept_greedy(a["target"], a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    h = _onehot(sv, a)
    _compare_onehot(h, oracle.spec_accept_onehot(a["target"], a["tokens"], a["parent"],
                                                 a["u_accept"], a["u_bonus"]), a)


def test_variants_status_and_edges(sv):
    a = _case(5, 4, 7, 100)
    a["parent"][1, 3] = 5          # not BFS
    a["tokens"][2, 4] = 100        # outside the vocabulary
    a["parent"][3] = [-1, 0, 1, 2, 3, 4, 5]   # a chain
    a["tokens"][3, 1:] = 7         # duplicate tokens along it
    for run, ref in ((_greedy, lambda: oracle.spec_accept_greedy(a["target"], a["tokens"],
                                                                  a["parent"])),
                     (_onehot, lambda: oracle.spec_accept_onehot(**a))):
        gpu = run(sv, a)
        orc = ref()
        assert gpu["status"].tolist() == orc["status"].tolist() == [0, 1, 2, 0]
        for b in (1, 2):
            assert (gpu["path"][b] == -1).all() and (gpu["out_tokens"][b] == -1).all()
            assert gpu["accept_len"][b] == 0
        for b in (0, 3):
            assert gpu["path"][b].tolist() == orc["path"][b].tolist()
    # a single-node tree: only the bonus token
    one = _case(6, 3, 1, 50)
    g = _greedy(sv, one)
    assert g["out_tokens"][:, 0].tolist() == np.argmax(one["target"][:, 0], -1).tolist()
    h = _onehot(sv, one)
    o = oracle.spec_accept_onehot(**one)
    _compare_onehot(h, o, one)


def test_onehot_lossless_on_gpu(sv):
    """Depth-1 tree with three fixed candidates (the draft's top-3): over 10^6
    sequences the emitted token follows the target softmax."""
    rng = np.random.default_rng(8)
    V, T = 8, 1_000_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    top3 = np.argsort(-q)[:3]
    tgt = np.broadcast_to(np.log(p).astype(np.float32), (T, 4, V))
    a = dict(target=tgt, tokens=np.broadcast_to(np.concatenate([[0], top3]).astype(np.int32), (T, 4)),
             parent=np.broadcast_to(np.array([-1, 0, 0, 0], np.int32), (T, 4)),
             u_accept=rng.random((T, 4), dtype=np.float32), u_bonus=rng.random(T, dtype=np.float32))
    gpu = _onehot(sv, a)
    counts = np.bincount(gpu["out_tokens"][:, 0], minlength=V)
    _, pval = chisquare(counts, p * T)
    assert pval > 1e-4, pval


def _bf16(x):
    """Logits rounded to bf16 on the CPU: the bf16 device tensor and the same
    values widened to float32 for the oracle."""
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    return t.cuda(), t.float().numpy()


BF16_VOCABS = [37, 4096, 5003, 32000, 128256]


@pytest.mark.parametrize("V", BF16_VOCABS)
def test_greedy_bf16_matches_oracle(sv, V):
    """bf16 rows: many equal maxima after rounding, each resolved to the
    lowest id on both sides."""
    B = 24 if V > 100000 else 48
    a = _case(V + 11, B, 15, V, noise=0.5)
    tb, tf = _bf16(a["target"])
    r = sv.spec_accept_greedy(tb, _dev(a["tokens"]), _dev(a["parent"]))
    torch.cuda.synchronize()
    gpu = {k: _np(v) for k, v in r.items()}
    orc = oracle.spec_accept_greedy(tf, a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(gpu[k], orc[k], err_msg=k)


@pytest.mark.parametrize("V", BF16_VOCABS)
def test_onehot_bf16_matches_oracle(sv, V):
    B = 24 if V > 100000 else 48
    a = _case(V + 13, B, 15, V, sigma=2.0 if V <= 5003 else 8.0, noise=0.7)
    tb, tf = _bf16(a["target"])
    r = sv.spec_accept_onehot(tb, _dev(a["tokens"]), _dev(a["parent"]), _dev(a["u_accept"]),
                              _dev(a["u_bonus"]))
    torch.cuda.synchronize()
    gpu = {k: _np(v) for k, v in r.items()}
    orc = oracle.spec_accept_onehot(tf, a["tokens"], a["parent"], a["u_accept"], a["u_bonus"])
    _compare_onehot(gpu, orc, dict(a, target=tf))


@pytest.mark.parametrize("V", [300000, 524288])
def test_variants_bf16_streaming_vocabularies(sv, V):
    a = _case(V + 17, 4, 15, V, sigma=8.0, noise=0.7)
    tb, tf = _bf16(a["target"])
    g = sv.spec_accept_greedy(tb, _dev(a["tokens"]), _dev(a["parent"]))
    h = sv.spec_accept_onehot(tb, _dev(a["tokens"]), _dev(a["parent"]), _dev(a["u_accept"]),
                              _dev(a["u_bonus"]))
    torch.cuda.synchronize()
    o = oracle.spec_accept_greedy(tf, a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens", "status"):
        np.testing.assert_array_equal(_np(g[k]), o[k], err_msg=k)
    _compare_onehot({k: _np(v) for k, v in h.items()},
                    oracle.spec_accept_onehot(tf, a["tokens"], a["parent"], a["u_accept"],
                                              a["u_bonus"]), dict(a, target=tf))


def test_variants_bf16_many_sequences(sv):
    a = _case(101, 64, 31, 128256, noise=1.5, binary=True)
    tb, tf = _bf16(a["target"])
    g = sv.spec_accept_greedy(tb, _dev(a["tokens"]), _dev(a["parent"]))
    h = sv.spec_accept_onehot(tb, _dev(a["tokens"]), _dev(a["parent"]), _dev(a["u_accept"]),
                              _dev(a["u_bonus"]))
    torch.cuda.synchronize()
    o = oracle.spec_accept_greedy(tf, a["tokens"], a["parent"])
    for k in ("accept_len", "path", "out_tokens"):
        np.testing.assert_array_equal(_np(g[k]), o[k], err_msg=k)
    _compare_onehot({k: _np(v) for k, v in h.items()},
                    oracle.spec_accept_onehot(tf, a["tokens"], a["parent"], a["u_accept"],
                                              a["u_bonus"]), dict(a, target=tf))
