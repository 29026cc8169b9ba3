"""Plain fp64 CPU oracle for one-pass tree verification.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg call it; the product path never does. It shares
no code with the CUDA library. The arithmetic lives in ``oracle.c`` (plain C,
fp64, optional OpenMP); this module only builds it with gcc and marshals numpy
arrays.

Functions (the C file cites the passage each one follows):
  tree_mask(parent)                      -> anc [B,N,W] uint64, depth [B,N], status [B]
  tree_attn(q, k, v, seq_lens, parent, scale, rows=None) -> out [R,D] f64, lse [R] f64
  spec_accept(target, draft, tokens, parent, u_accept, u_bonus) -> dict
  kv_commit(k_cache, v_cache, page_table, seq_lens, path, accept_len, N) -> dict
  spec_accept_greedy(target, tokens, parent) -> dict
  eagle2_pool / eagle2_expand / eagle2_finalize: EAGLE-2 tree construction
  spec_accept_onehot(target, tokens, parent, u_accept, u_bonus) -> dict
  lm_head_logits(hidden, W)              -> logits [..., V] f64
  spec_accept_lmhead(hidden, W, draft, tokens, parent, u_accept, u_bonus) -> dict
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into _build/liboracle.so (IEEE fp64, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_tree_mask.argtypes = [P, I, I, P, P, P]
            lib.oracle_tree_mask.restype = I
            lib.oracle_tree_attn.argtypes = [P, P, P, I, P, P, I, I, I, I, I, ctypes.c_double,
                                             P, I, P, P]
            lib.oracle_tree_attn.restype = I
            lib.oracle_spec_accept.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P, P, P, P, P, P]
            lib.oracle_spec_accept.restype = I
            lib.oracle_kv_commit.argtypes = [P, P, I, I, ctypes.c_longlong, I, I, P, I, P, P, P,
                                             I, I, I, I, P, P, I, P, P]
            lib.oracle_kv_commit.restype = I
            lib.oracle_spec_accept_greedy.argtypes = [P, P, P, I, I, I, P, P, P, P]
            lib.oracle_spec_accept_greedy.restype = I
            lib.oracle_spec_accept_onehot.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, P, P, P]
            lib.oracle_spec_accept_onehot.restype = I
            lib.oracle_eagle2_expand.argtypes = [P, I, I, I, I, P, I, P, P, P, P, P, P, P]
            lib.oracle_eagle2_expand.restype = I
            lib.oracle_eagle2_finalize.argtypes = [I, I, P, P, P, P, P, I, P, P, P, P, P, P, P]
            lib.oracle_eagle2_finalize.restype = I
            lib.oracle_lm_head.argtypes = [P, P, I, I, I, P]
            lib.oracle_lm_head.restype = I
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = I
            lib.oracle_set_threads.argtypes = [I]
            lib.oracle_set_threads.restype = None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().oracle_max_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def tree_mask(parent):
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    if parent.ndim == 1:
        parent = parent[None]
    B, N = parent.shape
    W = max(1, (N + 63) // 64)
    anc = np.zeros((B, N, W), dtype=np.uint64)
    depth = np.zeros((B, N), dtype=np.int32)
    status = np.zeros((B,), dtype=np.int32)
    rc = _load().oracle_tree_mask(_p(parent), B, N, _p(anc), _p(depth), _p(status))
    assert rc == 0
    return anc, depth, status


def tree_attn(q, k, v, seq_lens, parent, scale=None, rows=None):
    """q [B,N,Hq,D]; k, v [B,Tcap,Hkv,D] logical order (all float32 values)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    B, N, Hq, D = q.shape
    Tcap, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is None:
        R = B * N * Hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        R = rows_arr.shape[0]
    out = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros((R,), dtype=np.float64)
    rc = _load().oracle_tree_attn(_p(q), _p(k), _p(v), Tcap, _p(seq_lens), _p(parent), B, N, Hq,
                                  Hkv, D, float(scale), _p(rows_arr), R, _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_tree_attn: bad arguments")
    return out, lse


def spec_accept(target, draft, tokens, parent, u_accept, u_bonus, probe_token=None):
    """Acceptance walk in fp64. ``probe_token`` [B] (optional, -1 = none) asks for
    the normalised CDF of the final distribution just before and through that
    token (``probe_cdf`` [B, 3]: before, through, u_bonus)."""
    target = np.ascontiguousarray(target, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32)
    u_bonus = np.ascontiguousarray(u_bonus, dtype=np.float32)
    B, N, V = target.shape
    assert draft.shape == (B, N, V) and tokens.shape == (B, N) and parent.shape == (B, N)
    assert u_accept.shape == (B, N) and u_bonus.shape == (B,)
    out = {
        "accept_len": np.zeros((B,), np.int32),
        "path": np.zeros((B, N), np.int32),
        "out_tokens": np.zeros((B, N), np.int32),
        "ratio": np.zeros((B, N), np.float64),
        "accept_margin": np.zeros((B, N), np.float64),
        "bonus_margin": np.zeros((B,), np.float64),
        "n_rejects": np.zeros((B,), np.int32),
        "status": np.zeros((B,), np.int32),
        "probe_cdf": np.full((B, 3), np.nan, np.float64),
    }
    if probe_token is not None:
        probe_token = np.ascontiguousarray(probe_token, dtype=np.int32)
        assert probe_token.shape == (B,)
    rc = _load().oracle_spec_accept(
        _p(target), _p(draft), _p(tokens), _p(parent), _p(u_accept), _p(u_bonus), B, N, V,
        _p(out["accept_len"]), _p(out["path"]), _p(out["out_tokens"]), _p(out["ratio"]),
        _p(out["accept_margin"]), _p(out["bonus_margin"]), _p(out["n_rejects"]), _p(out["status"]),
        _p(probe_token), _p(out["probe_cdf"]) if probe_token is not None else None)
    assert rc == 0
    return out


def kv_commit(k_cache, v_cache, page_table, seq_lens, path, accept_len, N, max_free=None):
    """Commit the accepted path's K/V in place on copies of the caches.

    k_cache, v_cache: [layers, num_pages, page_size, Hkv, D] (or without the
    layer axis) numpy arrays of 2- or 4-byte elements (bf16 as uint16). Returns
    a dict with the committed caches ``k``, ``v`` and ``new_seq_lens``,
    ``freed`` [B, max_free], ``n_freed``, ``status``."""
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    assert k.shape == v.shape and k.dtype == v.dtype and k.itemsize in (2, 4)
    shp = k.shape if k.ndim == 5 else (1,) + k.shape
    layers, num_pages, page_size, Hkv, D = shp
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    path = np.ascontiguousarray(path, dtype=np.int32)
    accept_len = np.ascontiguousarray(accept_len, dtype=np.int32)
    B, max_pages = page_table.shape
    assert path.shape == (B, N) and accept_len.shape == (B,) and seq_lens.shape == (B,)
    if max_free is None:
        max_free = (N + page_size - 1) // page_size
    out = {
        "new_seq_lens": np.zeros((B,), np.int32),
        "freed": np.zeros((B, max_free), np.int32),
        "n_freed": np.zeros((B,), np.int32),
        "status": np.zeros((B,), np.int32),
    }
    stride = num_pages * page_size * Hkv * D
    rc = _load().oracle_kv_commit(
        _p(k), _p(v), k.itemsize, layers, stride, num_pages, page_size, _p(page_table), max_pages,
        _p(seq_lens), _p(path), _p(accept_len), B, N, Hkv, D, _p(out["new_seq_lens"]),
        _p(out["freed"]), max_free, _p(out["n_freed"]), _p(out["status"]))
    if rc != 0:
        raise ValueError("oracle_kv_commit: bad arguments")
    out["k"] = k
    out["v"] = v
    return out


def _variant_inputs(target, tokens, parent):
    target = np.ascontiguousarray(target, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    B, N, V = target.shape
    assert tokens.shape == (B, N) and parent.shape == (B, N)
    return target, tokens, parent, B, N, V


def spec_accept_greedy(target, tokens, parent):
    """Temperature-0 acceptance: argmax matching along the tree."""
    target, tokens, parent, B, N, V = _variant_inputs(target, tokens, parent)
    out = {"accept_len": np.zeros((B,), np.int32), "path": np.zeros((B, N), np.int32),
           "out_tokens": np.zeros((B, N), np.int32), "status": np.zeros((B,), np.int32)}
    rc = _load().oracle_spec_accept_greedy(
        _p(target), _p(tokens), _p(parent), B, N, V, _p(out["accept_len"]), _p(out["path"]),
        _p(out["out_tokens"]), _p(out["status"]))
    assert rc == 0
    return out


def spec_accept_onehot(target, tokens, parent, u_accept, u_bonus):
    """The sampling rule with q = one-hot(candidate) for every child."""
    target, tokens, parent, B, N, V = _variant_inputs(target, tokens, parent)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32)
    u_bonus = np.ascontiguousarray(u_bonus, dtype=np.float32)
    assert u_accept.shape == (B, N) and u_bonus.shape == (B,)
    out = {"accept_len": np.zeros((B,), np.int32), "path": np.zeros((B, N), np.int32),
           "out_tokens": np.zeros((B, N), np.int32), "ratio": np.zeros((B, N), np.float64),
           "accept_margin": np.zeros((B, N), np.float64),
           "bonus_margin": np.zeros((B,), np.float64), "status": np.zeros((B,), np.int32)}
    rc = _load().oracle_spec_accept_onehot(
        _p(target), _p(tokens), _p(parent), _p(u_accept), _p(u_bonus), B, N, V,
        _p(out["accept_len"]), _p(out["path"]), _p(out["out_tokens"]), _p(out["ratio"]),
        _p(out["accept_margin"]), _p(out["bonus_margin"]), _p(out["status"]))
    assert rc == 0
    return out


def eagle2_pool(root_tokens, capacity):
    """A fresh node pool per sequence holding only the root (cid 0, value 1)."""
    root_tokens = np.asarray(root_tokens, dtype=np.int32)
    B = root_tokens.shape[0]
    pool = {"parent": np.full((B, capacity), -1, np.int32),
            "depth": np.zeros((B, capacity), np.int32),
            "token": np.full((B, capacity), -1, np.int32),
            "value": np.zeros((B, capacity), np.float64),
            "count": np.ones((B,), np.int32)}
    pool["token"][:, 0] = root_tokens
    pool["value"][:, 0] = 1.0
    return pool


def eagle2_expand(pool, rows, frontier, k):
    """One expansion round in place on ``pool``. rows [B, R, V] are the draft
    logits at the frontier nodes frontier [B, R] (cids, -1 padded at the end).
    Returns (next_frontier [B, k], select_gap [B])."""
    rows = np.ascontiguousarray(rows, dtype=np.float32)
    frontier = np.ascontiguousarray(frontier, dtype=np.int32)
    B, R, V = rows.shape
    C = pool["parent"].shape[1]
    nxt = np.zeros((B, k), np.int32)
    gap = np.zeros((B,), np.float64)
    rc = _load().oracle_eagle2_expand(_p(rows), B, R, V, k, _p(frontier), C, _p(pool["parent"]),
                                      _p(pool["depth"]), _p(pool["token"]), _p(pool["value"]),
                                      _p(pool["count"]), _p(nxt), _p(gap))
    if rc != 0:
        raise ValueError("oracle_eagle2_expand: bad arguments")
    return nxt, gap


def eagle2_finalize(pool, n_nodes):
    """Rerank the pool and flatten the kept subtree in BFS order."""
    B, C = pool["parent"].shape
    out = {"parent": np.zeros((B, n_nodes), np.int32), "token": np.zeros((B, n_nodes), np.int32),
           "value": np.zeros((B, n_nodes), np.float64), "cid": np.zeros((B, n_nodes), np.int32),
           "n_out": np.zeros((B,), np.int32), "cut_gap": np.zeros((B,), np.float64),
           "connected": np.zeros((B,), np.int32)}
    rc = _load().oracle_eagle2_finalize(
        B, C, _p(pool["parent"]), _p(pool["depth"]), _p(pool["token"]), _p(pool["value"]),
        _p(pool["count"]), n_nodes, _p(out["parent"]), _p(out["token"]), _p(out["value"]),
        _p(out["cid"]), _p(out["n_out"]), _p(out["cut_gap"]), _p(out["connected"]))
    if rc != 0:
        raise ValueError("oracle_eagle2_finalize: bad arguments")
    return out


def lm_head_logits(hidden, W):
    """Target logits from the LM head: hidden [..., H] (one state per tree
    node) times W [V, H] transposed, in fp64. bf16 inputs must arrive widened
    to float32 (exactly)."""
    hidden = np.ascontiguousarray(hidden, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    H = hidden.shape[-1]
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H] with H = hidden.shape[-1]")
    R = hidden.size // H
    out = np.zeros((R, V), np.float64)
    rc = _load().oracle_lm_head(_p(hidden), _p(W), R, H, V, _p(out))
    if rc != 0:
        raise ValueError("oracle_lm_head: bad arguments")
    return out.reshape(hidden.shape[:-1] + (V,))


def spec_accept_lmhead(hidden, W, draft, tokens, parent, u_accept, u_bonus):
    """The acceptance walk with the target rows produced by the LM head:
    hidden [B, N, H], W [V, H]. The logits are the fp64 products rounded to
    float32 (the walk's logits type); the walk is spec_accept's. Returns
    spec_accept's dict plus "target" (the float32 logits it used)."""
    target = lm_head_logits(hidden, W).astype(np.float32)
    out = spec_accept(target, draft, tokens, parent, u_accept, u_bonus)
    out["target"] = target
    return out
