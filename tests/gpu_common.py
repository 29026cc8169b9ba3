"""Helpers shared by the GPU parity tests: moving generated inputs to the
device, running the oracle on the same inputs, and comparing acceptance
results with the near-tie rule.

Near ties. The oracle decides in fp64, the kernels in fp32 (with fp64 sums
of fp32 partials). Where a decision sits closer to its threshold than the
kernels' rounding can resolve, both answers are correct; such decisions are
compared for validity, every other one bit for bit:
  * accept tests u*q(x) < p~(x): flagged when |u q - p~| / max(u q, p~) < 1e-4
    (the kernels' relative error on p(x), q(x) and the residual mass is
    ~1e-6, set by expf's 2-ulp bound and fp32 sums of 4-element lanes);
  * the bonus token: flagged when u*sum(p~) lies within delta of a knot of
    the CDF, delta = 2e-6 for a target softmax and 2e-5 for a residual (the
    residual p - c q, c <= rejections + 1, amplifies the per-element error by
    (1 + c)/S). A flagged bonus token must still satisfy
    C(k-1) - delta <= u <= C(k) + delta on the oracle's fp64 CDF.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from synth.gen import logical_kv, bf16_bits_to_f32

ACCEPT_REL_TIE = 1e-4
BONUS_DELTA_PURE = 2e-6
BONUS_DELTA_RESIDUAL = 2e-5


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def device_inputs(inp, dev="cuda"):
    w = inp.w
    if w.dtype == "bf16":
        q = bf16_tensor(inp.q, dev)
        k = bf16_tensor(inp.k_cache, dev) if inp.k_cache is not None else None
        v = bf16_tensor(inp.v_cache, dev) if inp.v_cache is not None else None
    else:
        q = torch.from_numpy(inp.q).to(dev)
        k = torch.from_numpy(inp.k_cache).to(dev) if inp.k_cache is not None else None
        v = torch.from_numpy(inp.v_cache).to(dev) if inp.v_cache is not None else None
    d = {
        "q": q, "k": k, "v": v,
        "page_table": torch.from_numpy(inp.page_table).to(dev),
        "seq_lens": torch.from_numpy(inp.seq_lens).to(dev),
        "parent": torch.from_numpy(inp.parent).to(dev),
        "tokens": torch.from_numpy(inp.tokens).to(dev),
        "u_accept": torch.from_numpy(inp.u_accept).to(dev),
        "u_bonus": torch.from_numpy(inp.u_bonus).to(dev),
    }
    if inp.target is not None:
        d["target"] = torch.from_numpy(inp.target).to(dev)
        d["draft"] = torch.from_numpy(inp.draft).to(dev)
    return d


def as_f32(x, dtype):
    return bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, np.float32)


def oracle_logical_kv(inp, bs):
    """Logical K, V [len(bs), Tcap, Hkv, D] float32 for sequences bs, regenerated."""
    w = inp.w
    T = inp.seq_lens[bs].astype(np.int64) + w.N
    Tcap = int(T.max())
    K = np.zeros((len(bs), Tcap, w.Hkv, w.D), np.float32)
    V = np.zeros_like(K)
    for n, b in enumerate(bs):
        for g in range(w.Hkv):
            kk, vv = logical_kv(w, inp.seed, int(b), g, int(T[n]))
            K[n, : T[n], g] = as_f32(kk, w.dtype)
            V[n, : T[n], g] = as_f32(vv, w.dtype)
    return K, V


def oracle_attention(inp, bs=None, rows=None):
    """Oracle attention for sequences bs (all when None); rows = (b_local, i, h) triples."""
    w = inp.w
    if bs is None:
        bs = np.arange(w.B)
    bs = np.asarray(bs)
    K, V = oracle_logical_kv(inp, bs)
    q = as_f32(inp.q[bs], w.dtype)
    out, lse = oracle.tree_attn(q, K, V, inp.seq_lens[bs], inp.parent[bs], rows=rows)
    return out, lse


def compare_accept(gpu: dict, inp_arrays: dict, orc: dict, max_flag_frac=0.05):
    """Bit-exact comparison of walk outputs except flagged near ties (validated).

    inp_arrays: numpy target, draft, tokens, parent, u_accept, u_bonus.
    Returns a dict of counts; raises AssertionError on any unflagged mismatch.
    """
    al = gpu["accept_len"]; path = gpu["path"]; out = gpu["out_tokens"]; st = gpu["status"]
    B, N = path.shape
    assert (st == orc["status"]).all(), "status differs"
    bonus_b, walk_b = [], []
    for b in range(B):
        if (al[b] == orc["accept_len"][b] and (path[b] == orc["path"][b]).all()
                and (out[b] == orc["out_tokens"][b]).all()):
            continue
        same_walk = al[b] == orc["accept_len"][b] and (path[b] == orc["path"][b]).all()
        if same_walk:
            bonus_b.append(b)
            continue
        am = orc["accept_margin"][b]
        tested = ~np.isnan(am)
        assert (am[tested] < ACCEPT_REL_TIE).any(), (
            f"sequence {b}: walk differs without a near tie: gpu path {path[b]} len {al[b]}, "
            f"oracle path {orc['path'][b]} len {orc['accept_len'][b]}")
        walk_b.append(b)
    if bonus_b:
        probe = np.full(B, -1, np.int32)
        for b in bonus_b:
            probe[b] = out[b, al[b]]
        o2 = oracle.spec_accept(inp_arrays["target"], inp_arrays["draft"], inp_arrays["tokens"],
                                inp_arrays["parent"], inp_arrays["u_accept"],
                                inp_arrays["u_bonus"], probe_token=probe)
        for b in bonus_b:
            delta = BONUS_DELTA_PURE if orc["n_rejects"][b] == 0 else BONUS_DELTA_RESIDUAL
            lo, hi, u = o2["probe_cdf"][b]
            assert orc["bonus_margin"][b] < delta, (
                f"sequence {b}: bonus token {out[b, al[b]]} vs oracle "
                f"{orc['out_tokens'][b, al[b]]} with margin {orc['bonus_margin'][b]:.3g}")
            assert lo - delta <= u <= hi + delta, (
                f"sequence {b}: gpu bonus token outside the CDF crossing: {lo} {u} {hi}")
    flagged = len(bonus_b) + len(walk_b)
    assert flagged <= max(2, math.ceil(max_flag_frac * B)), f"{flagged} near ties out of {B}"
    return {"bonus_near_ties": len(bonus_b), "walk_near_ties": len(walk_b), "B": B}


def compare_ratio(gpu_ratio, orc, rtol_first=1e-5, rtol_after=1e-3):
    """Ratios of nodes tested by both walks (same path), tolerance looser after
    a rejection where p - c q cancels."""
    r_o = orc["ratio"]
    same = (gpu_ratio is not None)
    if not same:
        return 0.0
    both = ~np.isnan(r_o) & ~np.isnan(gpu_ratio)
    if not both.any():
        return 0.0
    err = np.abs(gpu_ratio[both] - r_o[both]) / np.maximum(1.0, np.abs(r_o[both]))
    return float(err.max())
