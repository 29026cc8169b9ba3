"""Helpers shared by the GPU parity tests: moving generated inputs to the
device, running the oracle on the same inputs, and comparing acceptance
results decision by decision.

Parity bar for the acceptance walks. The oracle decides in fp64, the kernels
in fp32 (masses and CDF prefixes in double-float). Two walks are compared as
the ordered lists of their decisions (tested node, accepted or not) and their
bonus token. They must be identical, except that the FIRST differing decision
may differ when it lies within the kernels' rounding of its threshold, and a
bonus token may differ (on identical walks) when u*sum(p~) lies within the
kernels' rounding of a CDF knot. Everything else is bit for bit.

Error model, from the closed form of the residual after k rejected siblings
at the parent (c_0 = 0, S_0 = 1, c_{k+1} = c_k + S_k,
S_{k+1} = sum_v max(0, p_v - c_{k+1} q_v), and p~ = max(0, p - c q)/S): the
kernel tests L = u q(x) S against R = max(0, p(x) - c q(x)). With every
per-element probability accurate to a relative eps, |dq| <= eps q(x),
|dp| <= eps p(x) and |dS| <= eps (1 + c) (S sums p - c q over the positive
part, whose terms add up to at most 1 + c), so
    |dL - dR| <= eps * E,  E = L (1 + [k > 0] (1 + c)/S) + p(x) + c q(x).
A decision is a near tie when |L - R| <= TIE_TOL * E / 2, which at a first
test (k = 0) is |u q - p| <= TIE_TOL * (u q + p)/2 <= TIE_TOL * max(u q, p):
relative 1e-5. Ratios p~(x)/q(x) = R/(S q) of nodes that both walks tested
in the same state are held to
    |r_gpu - r| <= TIE_TOL * ((p(x) + c q(x))/(S q(x)) + r (1 + [k > 0] (1 + c)/S)) / 2,
which is 1e-5 relative at a first test. The bonus token at a node with k
rejections may differ when u*sum(p~) lies within
BONUS_DELTA * (1 + c)/S of a knot of the oracle's normalised CDF (the
residual's per-element error grows by (1 + c)/S), and the GPU's token must
then still satisfy C(k-1) - delta <= u <= C(k) + delta on that CDF.

Every comparison appends its counts (sequences, decisions compared, ties
taken, largest ratio error against its bound) as one JSON line to the file
named by the environment variable SVF_PARITY_LOG, when it is set.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from synth.gen import logical_kv, bf16_bits_to_f32

TIE_TOL = 1e-5
BONUS_DELTA = 2e-6
MAX_TIE_FRAC = 0.01


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


# ---------------------------------------------------------------------------
# acceptance comparisons
# ---------------------------------------------------------------------------

def log_parity(record: dict) -> None:
    """Append one comparison's counts to $SVF_PARITY_LOG (if set)."""
    path = os.environ.get("SVF_PARITY_LOG")
    if not path:
        return
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], **record}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def softmax64(row) -> np.ndarray:
    r = np.asarray(row, np.float64)
    e = np.exp(r - r.max())
    return e / e.sum()


def residual_state(p: np.ndarray, q: np.ndarray, k: int):
    """(c_k, S_k) of the closed-form residual after k rejections (fp64)."""
    c, S = 0.0, 1.0
    for _ in range(k):
        c = c + S
        S = float(np.maximum(0.0, p - c * q).sum())
        if S <= 0.0:
            break
    return c, S


def decisions(parent_b, ratio_b, path_b, alen_b):
    """Ordered decisions of one finished walk: (node, parent, prior rejections
    among its siblings, accepted). A node is tested iff its ratio is not NaN."""
    out = []
    N = len(parent_b)
    steps = [int(x) for x in path_b[: int(alen_b) + 1]]
    for i, j in enumerate(steps):
        nxt = steps[i + 1] if i + 1 < len(steps) else -1
        k = 0
        for c in range(j + 1, N):
            if parent_b[c] != j or np.isnan(ratio_b[c]):
                continue
            acc = c == nxt
            out.append((c, j, k, acc))
            if acc:
                break
            k += 1
    return out


class _Rows:
    """fp64 softmax rows of one sequence, computed on demand."""

    def __init__(self, target_b, draft_b):
        self.t, self.d = target_b, draft_b
        self.cache = {}

    def pq(self, j):
        if j not in self.cache:
            self.cache[j] = (softmax64(self.t[j]), softmax64(self.d[j]))
        return self.cache[j]


def _tie_scale(rows, tokens_b, u_b, c_node, j, k):
    """(|L - R|, E) of the test of node c_node at parent j after k rejections."""
    p, q = rows.pq(j)
    c, S = residual_state(p, q, k)
    x = int(tokens_b[c_node])
    u = float(u_b[c_node])
    L = u * q[x] * S
    R = max(0.0, p[x] - c * q[x])
    E = L * (1.0 + ((1.0 + c) / S if k > 0 else 0.0)) + p[x] + c * q[x]
    return abs(L - R), E


def compare_accept(gpu: dict, inp_arrays: dict, orc: dict, max_tie_frac=MAX_TIE_FRAC,
                   tie_tol=TIE_TOL, bonus_delta=BONUS_DELTA):
    """Decision-by-decision comparison of a GPU walk with the oracle's.

    inp_arrays: numpy target, draft, tokens, parent, u_accept, u_bonus.
    ``tie_tol`` is the per-element relative error eps of the model above
    (1e-5 for logits both sides read exactly; larger where the GPU's logits
    carry their own rounding, as when an LM head produced them).
    Returns a dict of counts; raises AssertionError on any mismatch that is
    not a near tie under the error model of this module."""
    al = gpu["accept_len"]; path = gpu["path"]; out = gpu["out_tokens"]; st = gpu["status"]
    B, N = path.shape
    assert (st == orc["status"]).all(), "status differs"
    tgt, dft = inp_arrays["target"], inp_arrays["draft"]
    par, tok, ua = inp_arrays["parent"], inp_arrays["tokens"], inp_arrays["u_accept"]
    g_ratio = gpu.get("ratio")
    walk_b, bonus_b = [], []
    n_dec = 0
    ratio_worst = 0.0   # largest |r_gpu - r| / bound over nodes tested in the same state
    ratio_first = 0.0   # largest relative error at first tests
    for b in range(B):
        if st[b] != 0:
            assert (path[b] == orc["path"][b]).all() and al[b] == orc["accept_len"][b]
            continue
        o_dec = decisions(par[b], orc["ratio"][b], orc["path"][b], orc["accept_len"][b])
        n_dec += len(o_dec)
        same_walk = al[b] == orc["accept_len"][b] and (path[b] == orc["path"][b]).all()
        rows = None
        if g_ratio is not None:
            g_dec = decisions(par[b], g_ratio[b], path[b], al[b])
            first = next((i for i, (a, c) in enumerate(zip(o_dec, g_dec)) if a != c),
                         None if len(o_dec) == len(g_dec) else min(len(o_dec), len(g_dec)))
            # ratios of the decisions both walks took in the same state
            upto = len(o_dec) if first is None else first
            if upto:
                rows = _Rows(tgt[b], dft[b])
            for (c, j, k, _) in o_dec[:upto]:
                p, q = rows.pq(j)
                cc, S = residual_state(p, q, k)
                x = int(tok[b, c])
                r = orc["ratio"][b, c]
                bound = tie_tol * ((p[x] + cc * q[x]) / (S * q[x])
                                   + r * (1.0 + ((1.0 + cc) / S if k > 0 else 0.0))) / 2
                err = abs(float(g_ratio[b, c]) - r)
                ratio_worst = max(ratio_worst, err / bound)
                if k == 0:
                    ratio_first = max(ratio_first, err / r)
                assert err <= bound, (
                    f"sequence {b} node {c}: ratio {g_ratio[b, c]} vs {r} (k={k}, bound {bound:.3g})")
        else:
            first = None if same_walk else 0
        if same_walk and first is None:
            if (out[b] == orc["out_tokens"][b]).all():
                continue
            bonus_b.append(b)
            continue
        # the walks part: the first differing decision must be a near tie
        assert first is not None and first < len(o_dec), (
            f"sequence {b}: walks differ with no differing oracle decision")
        c, j, k, _ = o_dec[first]
        if rows is None:
            rows = _Rows(tgt[b], dft[b])
        gap, E = _tie_scale(rows, tok[b], ua[b], c, j, k)
        assert gap <= tie_tol * E / 2, (
            f"sequence {b}: walk differs at node {c} without a near tie (gap {gap:.3g}, "
            f"scale {E:.3g}): gpu path {path[b]} len {al[b]}, oracle path {orc['path'][b]} "
            f"len {orc['accept_len'][b]}")
        walk_b.append(b)
    if bonus_b:
        probe = np.full(B, -1, np.int32)
        for b in bonus_b:
            probe[b] = out[b, al[b]]
        o2 = oracle.spec_accept(tgt, dft, tok, par, ua, inp_arrays["u_bonus"], probe_token=probe)
        for b in bonus_b:
            k = int(orc["n_rejects"][b])
            amp = 1.0
            if k > 0:
                j = int(orc["path"][b, orc["accept_len"][b]])
                p, q = softmax64(tgt[b, j]), softmax64(dft[b, j])
                cc, S = residual_state(p, q, k)
                amp = (1.0 + cc) / S
            delta = bonus_delta * amp
            lo, hi, u = o2["probe_cdf"][b]
            assert orc["bonus_margin"][b] < delta, (
                f"sequence {b}: bonus token {out[b, al[b]]} vs oracle "
                f"{orc['out_tokens'][b, al[b]]} with margin {orc['bonus_margin'][b]:.3g} "
                f"(delta {delta:.3g})")
            assert lo - delta <= u <= hi + delta, (
                f"sequence {b}: gpu bonus token outside the CDF crossing: {lo} {u} {hi}")
    ties = len(bonus_b) + len(walk_b)
    stats = {"B": B, "decisions": n_dec, "walk_ties": len(walk_b), "bonus_ties": len(bonus_b),
             "ratio_err_over_bound": ratio_worst, "ratio_rel_err_first_tests": ratio_first}
    log_parity({"kind": "spec_accept", **stats})
    assert ties <= max(1, math.ceil(max_tie_frac * B)), f"{ties} near ties out of {B}"
    return stats


def onehot_decisions(parent_b, ratio_b, path_b, alen_b):
    return decisions(parent_b, ratio_b, path_b, alen_b)


def compare_onehot(gpu: dict, target: np.ndarray, tokens: np.ndarray, parent: np.ndarray,
                   u_accept: np.ndarray, orc: dict, max_tie_frac=MAX_TIE_FRAC):
    """One-hot candidates: q = one-hot(x) per child, so a test is u < p~(x)
    with p~(x) = p(x)/(1 - p(Rj)) after rejecting the distinct tokens Rj.
    Error model: L = u (1 - p(Rj)), R = p(x); |dL - dR| <= eps (u p(Rj) + p(x)
    + [k > 0] u); a near tie is |L - R| <= TIE_TOL * (L + u p(Rj) + p(x))/2
    (relative 1e-5 at a first test). Ratios (= p~(x)) are held to
    TIE_TOL * r * (1 + p(Rj)/(1 - p(Rj))). A differing bonus token needs the
    oracle's margin below BONUS_DELTA / (1 - p(Rj))."""
    B = gpu["path"].shape[0]
    assert (gpu["status"] == orc["status"]).all()
    ties = 0
    n_dec = 0
    worst = 0.0
    for b in range(B):
        if gpu["status"][b] != 0:
            continue
        o_dec = decisions(parent[b], orc["ratio"][b], orc["path"][b], orc["accept_len"][b])
        g_dec = decisions(parent[b], gpu["ratio"][b], gpu["path"][b], gpu["accept_len"][b])
        n_dec += len(o_dec)
        first = next((i for i, (a, c) in enumerate(zip(o_dec, g_dec)) if a != c),
                     None if len(o_dec) == len(g_dec) else min(len(o_dec), len(g_dec)))
        upto = len(o_dec) if first is None else first
        cache = {}

        def p_of(j):
            if j not in cache:
                cache[j] = softmax64(target[b, j])
            return cache[j]

        def removed(c, j):
            """Mass of the distinct tokens of c's earlier siblings (all rejected)."""
            p = p_of(j)
            toks = {int(tokens[b, s]) for s in range(j + 1, c) if parent[b, s] == j}
            return float(sum(p[t] for t in toks))

        for (c, j, k, _) in o_dec[:upto]:
            pr = removed(c, j)
            r = orc["ratio"][b, c]
            bound = TIE_TOL * r * (1.0 + pr / max(1e-300, 1.0 - pr))
            err = abs(float(gpu["ratio"][b, c]) - r)
            worst = max(worst, err / max(bound, 1e-300))
            assert err <= bound or err < 1e-12, (
                f"sequence {b} node {c}: ratio {gpu['ratio'][b, c]} vs {r} (bound {bound:.3g})")
        if first is None:
            if (gpu["out_tokens"][b] == orc["out_tokens"][b]).all():
                continue
            j = int(orc["path"][b, orc["accept_len"][b]])
            kids = [s for s in range(j + 1, len(parent[b])) if parent[b, s] == j]
            pr = removed(kids[-1] + 1 if kids else j + 1, j) if kids else 0.0
            delta = BONUS_DELTA / max(1e-300, 1.0 - pr)
            assert orc["bonus_margin"][b] < delta, (
                f"sequence {b}: bonus {gpu['out_tokens'][b]} vs {orc['out_tokens'][b]}, "
                f"margin {orc['bonus_margin'][b]:.3g} (delta {delta:.3g})")
            ties += 1
            continue
        assert first < len(o_dec), f"sequence {b}: walks differ with no differing oracle decision"
        c, j, k, _ = o_dec[first]
        pr = removed(c, j)
        p = p_of(j)
        x = int(tokens[b, c])
        u = float(u_accept[b, c])
        L, R = u * (1.0 - pr), float(p[x])
        E = L + u * pr + R + (u if k > 0 else 0.0)
        assert abs(L - R) <= TIE_TOL * E / 2, (
            f"sequence {b}: path {gpu['path'][b]} vs {orc['path'][b]} at node {c}, gap "
            f"{abs(L - R):.3g}")
        ties += 1
    log_parity({"kind": "spec_accept_onehot", "B": B, "decisions": n_dec, "ties": ties,
                "ratio_err_over_bound": worst})
    assert ties <= max(1, math.ceil(max_tie_frac * B)), f"{ties} near ties out of {B}"
    return ties
