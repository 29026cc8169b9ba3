"""GPU parity of svf_kv_commit against the oracle: the whole cache, the new
lengths, the freed pages and the status words must match bit for bit."""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bf16_tensor
from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


def _np(t):
    return t.detach().cpu().numpy()


def _random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)


def _root_path(parent, node):
    p = []
    while node != -1:
        p.append(int(node))
        node = int(parent[node])
    return p[::-1]


def _paths(rng, parent, full=False):
    """A random accepted path per sequence: a prefix of a root path."""
    B, N = parent.shape
    path = np.full((B, N), -1, np.int32)
    alen = np.zeros(B, np.int32)
    for b in range(B):
        p = _root_path(parent[b], int(rng.integers(0, N)))
        if not full:
            p = p[: int(rng.integers(1, len(p) + 1))]
        path[b, : len(p)] = p
        alen[b] = len(p) - 1
    return path, alen


def _cache(rng, layers, num_pages, ps, Hkv, D, dtype):
    shape = (layers, num_pages, ps, Hkv, D)
    if dtype == "bf16":
        return (rng.integers(0, 1 << 16, size=shape, dtype=np.uint16),
                rng.integers(0, 1 << 16, size=shape, dtype=np.uint16))
    x = rng.standard_normal(shape).astype(np.float32)
    return x, rng.standard_normal(shape).astype(np.float32)


def _to_dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _from_dev(t, dtype):
    if dtype == "bf16":
        return _np(t.view(torch.int16)).view(np.uint16)
    return _np(t)


def _table(rng, lens, N, ps, spare=2):
    need = [-(-(int(L) + N) // ps) for L in lens]
    num_pages = sum(need) + spare
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((len(lens), max(need) + 1), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at: at + n]
        at += n
    return table, num_pages


def _run(sv, k, v, table, lens, path, alen, dtype, max_free=None):
    kd, vd = _to_dev(k, dtype), _to_dev(v, dtype)
    if k.shape[0] == 1 and np.random.default_rng(int(lens.sum())).integers(0, 2):
        kd, vd = kd[0], vd[0]          # the single-layer form without the layer axis
    res = sv.kv_commit(kd, vd, torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                       torch.from_numpy(path).cuda(), torch.from_numpy(alen).cuda(),
                       max_free=max_free)
    torch.cuda.synchronize()
    out = {n: _np(t) for n, t in res.items()}
    out["k"] = _from_dev(kd, dtype).reshape(k.shape)
    out["v"] = _from_dev(vd, dtype).reshape(v.shape)
    return out


def _compare(gpu, orc, max_free):
    for n in ("new_seq_lens", "n_freed", "status"):
        np.testing.assert_array_equal(gpu[n], orc[n], err_msg=n)
    np.testing.assert_array_equal(gpu["freed"][:, :max_free], orc["freed"], err_msg="freed")
    np.testing.assert_array_equal(gpu["k"], orc["k"])
    np.testing.assert_array_equal(gpu["v"], orc["v"])


CASES = [
    # B, N, ps, layers, Hkv, D, dtype, max prefix
    (1, 31, 16, 1, 8, 128, "bf16", 2048),
    (4, 60, 16, 2, 8, 128, "bf16", 300),
    (5, 64, 1, 1, 2, 64, "bf16", 40),
    (3, 17, 4, 3, 2, 64, "f32", 50),
    (7, 9, 64, 1, 4, 128, "f32", 500),
    (2, 1, 16, 1, 8, 128, "bf16", 33),
    (2, 200, 32, 1, 1, 64, "bf16", 70),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}N{c[1]}ps{c[2]}l{c[3]}{c[6]}" for c in CASES])
@pytest.mark.parametrize("full", [False, True])
def test_commit_matches_oracle(sv, case, full):
    B, N, ps, layers, Hkv, D, dtype, lmax = case
    rng = np.random.default_rng(2 * CASES.index(case) + int(full))
    lens = rng.integers(0, lmax + 1, size=B).astype(np.int32)
    table, num_pages = _table(rng, lens, N, ps)
    k, v = _cache(rng, layers, num_pages, ps, Hkv, D, dtype)
    parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    path, alen = _paths(rng, parent, full)
    max_free = -(-N // ps)
    gpu = _run(sv, k, v, table, lens, path, alen, dtype, max_free)
    orc = oracle.kv_commit(k, v, table, lens, path, alen, N, max_free)
    _compare(gpu, orc, max_free)


def test_commit_chain_and_root_only(sv):
    rng = np.random.default_rng(5)
    B, N, ps = 4, 16, 16
    lens = np.array([0, 15, 16, 1000], np.int32)
    table, num_pages = _table(rng, lens, N, ps)
    k, v = _cache(rng, 1, num_pages, ps, 8, 128, "bf16")
    path = np.full((B, N), -1, np.int32)
    alen = np.array([0, 15, 7, 3], np.int32)
    for b in range(B):
        path[b, : alen[b] + 1] = np.arange(alen[b] + 1)
    gpu = _run(sv, k, v, table, lens, path, alen, "bf16")
    orc = oracle.kv_commit(k, v, table, lens, path, alen, N)
    _compare(gpu, orc, 1)
    np.testing.assert_array_equal(gpu["k"], k)  # a chain is already in place


def test_commit_status_mix(sv):
    """Bad sequences are flagged and left alone; the good ones in the same call
    are committed."""
    rng = np.random.default_rng(6)
    B, N, ps = 6, 12, 4
    lens = np.array([3, 9, 4, 0, 7, 2], np.int32)
    table, num_pages = _table(rng, lens, N, ps)
    k, v = _cache(rng, 2, num_pages, ps, 2, 64, "bf16")
    parent = np.stack([_random_tree(rng, N) for _ in range(B)])
    path, alen = _paths(rng, parent, full=True)
    alen[1] = N                       # accept_len out of range
    path[2, 0] = 3                    # the path does not start at the root
    if alen[3] >= 1:
        path[3, 1] = 0                # not increasing
    else:
        alen[3] = -1
    table[4, 1] = num_pages + 5       # a page outside the cache
    lens[5] = table.shape[1] * ps     # past the page table
    gpu = _run(sv, k, v, table, lens, path, alen, "bf16")
    orc = oracle.kv_commit(k, v, table, lens, path, alen, N)
    assert orc["status"].tolist()[1:] == [32, 32, 32, 4, 8]
    _compare(gpu, orc, -(-N // ps))


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_commit_workloads_full(sv, idx):
    """The benchmark workloads' caches (one layer), random accepted paths of
    their trees, against the oracle over the whole cache."""
    w = WORKLOADS[idx]
    inp = make_inputs(w, 1000 + idx, with_kv=True, with_logits=False)
    rng = np.random.default_rng(idx)
    path, alen = _paths(rng, inp.parent, full=True)
    k, v = inp.k_cache[None], inp.v_cache[None]
    gpu = _run(sv, k, v, inp.page_table, inp.seq_lens, path, alen, "bf16")
    orc = oracle.kv_commit(k, v, inp.page_table, inp.seq_lens, path, alen, w.N)
    _compare(gpu, orc, -(-w.N // inp.page_size))


def test_commit_serving_70b_sampled(sv):
    """Full-size 70B-shaped paged cache (8.6 GB): every committed row must be
    the pre-commit row of its path node; sampled other rows are unchanged."""
    w = WORKLOADS[4]
    inp = make_inputs(w, 1004, with_kv=True, with_logits=False)
    rng = np.random.default_rng(4)
    path, alen = _paths(rng, inp.parent, full=True)
    kd, vd = bf16_tensor(inp.k_cache, "cuda"), bf16_tensor(inp.v_cache, "cuda")
    res = sv.kv_commit(kd, vd, torch.from_numpy(inp.page_table).cuda(),
                       torch.from_numpy(inp.seq_lens).cuda(), torch.from_numpy(path).cuda(),
                       torch.from_numpy(alen).cuda())
    torch.cuda.synchronize()
    assert (_np(res["status"]) == 0).all()
    np.testing.assert_array_equal(_np(res["new_seq_lens"]), inp.seq_lens + alen + 1)
    ps = inp.page_size
    kb = kd.view(torch.int16)
    vb = vd.view(torch.int16)

    def rows(cache_bits, b, toks):
        toks = np.asarray(toks)
        pages = inp.page_table[b, toks // ps]
        return _np(cache_bits[torch.from_numpy(pages).cuda().long(),
                              torch.from_numpy(toks % ps).cuda().long()]).view(np.uint16)

    for b in range(w.B):
        L, n = int(inp.seq_lens[b]), int(alen[b]) + 1
        src = L + path[b, :n]
        pages = inp.page_table[b, src // ps]
        np.testing.assert_array_equal(rows(kb, b, L + np.arange(n)), inp.k_cache[pages, src % ps])
        np.testing.assert_array_equal(rows(vb, b, L + np.arange(n)), inp.v_cache[pages, src % ps])
        other = np.concatenate([rng.integers(0, L, size=8), L + np.arange(n, w.N)])
        pages = inp.page_table[b, other // ps]
        np.testing.assert_array_equal(rows(kb, b, other), inp.k_cache[pages, other % ps])
