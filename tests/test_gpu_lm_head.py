"""GPU parity of the LM head (target logits from hidden states) and of the
acceptance walk fed by it, against the oracle.

Logits: every element within the fp32 rounding bound of the tensor cores'
accumulation, |l_gpu - l| <= (H/16 + 16) * 2^-24 * sum_k |h_k W_vk|: one
rounding of the accumulator per 16-element MMA step plus slack for the
rounding inside a step. The walk fed by the GPU's logits is compared with the
oracle's walk on the oracle's logits decision by decision; its near-tie
tolerance is the per-element probability error those logits allow,
2 max|l_gpu - l| (a softmax probability moves by at most the largest logit
change twice), and never below the 1e-5 of the plain walk.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import BONUS_DELTA, TIE_TOL, compare_accept, log_parity, softmax64
from synth.gen import f32_to_bf16_bits, bf16_bits_to_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


def _bf16(rng, shape, sigma):
    """bf16 bit patterns of N(0, sigma^2) draws and their exact float32 values."""
    x = (sigma * rng.standard_normal(int(np.prod(shape)), dtype=np.float32)).reshape(shape)
    bits = f32_to_bf16_bits(x)
    return bits, bf16_bits_to_f32(bits)


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bound(h, W, H):
    """The accumulation bound of every (row, vocabulary) element (fp64 result;
    the sums of magnitudes in blocks of vocabulary rows)."""
    ha = np.abs(h.astype(np.float64))
    out = np.empty((h.shape[0], W.shape[0]), np.float64)
    for v0 in range(0, W.shape[0], 8192):
        out[:, v0:v0 + 8192] = ha @ np.abs(W[v0:v0 + 8192].astype(np.float64)).T
    return (H / 16 + 16) * 2.0 ** -24 * out


def _case(seed, R, H, V):
    rng = np.random.default_rng(seed)
    hb, hf = _bf16(rng, (R, H), 1.0)
    wb, wf = _bf16(rng, (V, H), 3.0 / np.sqrt(H))   # logits ~ N(0, 3^2)
    return hb, hf, wb, wf


# (R, H, V): a binary tree at batch 1; odd sizes (V not a multiple of 128, R
# not a multiple of 32); the EAGLE-2 batch at the 128K vocabulary; the
# multicast path (R >= 512) with an odd tile width; the 70B serving shape;
# a vocabulary past 2^18 with a ragged last tile, and 313 weight tiles at 200
# rows (a second wave of 9 tiles).
LM_CASES = [
    (31, 4096, 32000, None),
    (7, 128, 300001, None),
    (200, 192, 40000, None),
    (60, 256, 1000, None),
    (1000, 64, 300, None),
    (240, 4096, 128256, 6),
    (600, 128, 5000, None),
    (1984, 1024, 32000, 8),
    (1984, 8192, 128256, 4),
]


@pytest.mark.parametrize("R,H,V,sample", LM_CASES)
def test_lm_head_matches_oracle(sv, R, H, V, sample):
    hb, hf, wb, wf = _case(R + V + H, R, H, V)
    logits = sv.lm_head(_dev_bf16(hb), _dev_bf16(wb))
    torch.cuda.synchronize()
    g = logits.cpu().numpy()
    rows = np.arange(R) if sample is None else np.unique(
        np.concatenate([[0, R - 1], np.random.default_rng(R).integers(0, R, sample - 2)]))
    ref = oracle.lm_head_logits(hf[rows], wf)
    bound = _bound(hf[rows], wf, H)
    err = np.abs(g[rows].astype(np.float64) - ref)
    worst = float((err / bound).max())
    log_parity({"kind": "lm_head", "R": R, "H": H, "V": V, "rows": int(len(rows)),
                "max_abs_err": float(err.max()), "err_over_bound": worst})
    print(f"R={R} H={H} V={V}: max|err| {err.max():.3g}, err/bound {worst:.3g}")
    assert worst <= 1.0


def test_lm_head_rows_past_the_batch_are_untouched(sv):
    """The call writes exactly [R, V]: a sentinel after the last row survives."""
    R, H, V = 33, 128, 515
    hb, hf, wb, wf = _case(9, R, H, V)
    buf = torch.full((R + 1, V), 7.0, dtype=torch.float32, device="cuda")
    sv.lm_head(_dev_bf16(hb), _dev_bf16(wb), logits=buf[:R])
    torch.cuda.synchronize()
    assert bool((buf[R] == 7.0).all())
    ref = oracle.lm_head_logits(hf, wf)
    assert (np.abs(buf[:R].cpu().numpy() - ref) <= _bound(hf, wf, H)).all()


def _binary_parent(n):
    p = (np.arange(n) - 1) // 2
    p[0] = -1
    return p.astype(np.int32)


@pytest.mark.parametrize("B,N,H,V", [(1, 31, 4096, 32000), (4, 15, 4096, 128256),
                                     (16, 7, 512, 1000)])
def test_spec_accept_lmhead_matches_oracle(sv, B, N, H, V):
    rng = np.random.default_rng(B * 1000 + N)
    hb, hf = _bf16(rng, (B, N, H), 1.0)
    wb, wf = _bf16(rng, (V, H), 3.0 / np.sqrt(H))
    parent = np.broadcast_to(_binary_parent(N), (B, N)).copy()
    # the drafter's rows: the oracle's target rows plus noise; the children of
    # a node carry its draft's top tokens, as in the binary-tree workloads
    t_ref = oracle.lm_head_logits(hf, wf).astype(np.float32)
    draft = (t_ref + 1.5 * rng.standard_normal((B, N, V), dtype=np.float32)).astype(np.float32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for j in range(N):
            kids = [c for c in (2 * j + 1, 2 * j + 2) if c < N]
            if kids:
                order = np.lexsort((np.arange(V), -softmax64(draft[b, j])))[: len(kids)]
                tokens[b, kids] = order
    u_acc = rng.random((B, N), dtype=np.float32)
    u_bon = rng.random(B, dtype=np.float32)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    res = sv.spec_accept_lmhead(_dev_bf16(hb), _dev_bf16(wb), d(draft), d(tokens), d(parent),
                                d(u_acc), d(u_bon))
    torch.cuda.synchronize()
    assert int(res["lm_status"].item()) == 0
    g_logits = res["target_logits"].cpu().numpy()
    orc = oracle.spec_accept_lmhead(hf, wf, draft, tokens, parent, u_acc, u_bon)
    err = np.abs(g_logits.astype(np.float64) - oracle.lm_head_logits(hf, wf))
    assert (err <= _bound(hf.reshape(B * N, H), wf, H).reshape(B, N, V)).all()
    # the fused call's walk is svf_spec_accept's on the same logits
    plain = sv.spec_accept(res["target_logits"], d(draft), d(tokens), d(parent), d(u_acc),
                           d(u_bon))
    torch.cuda.synchronize()
    for k in ("accept_len", "path", "out_tokens", "status"):
        assert torch.equal(plain[k], res[k]), k
    gpu = {k: res[k].cpu().numpy() for k in ("accept_len", "path", "out_tokens", "ratio",
                                              "status")}
    arrs = dict(target=orc["target"], draft=draft, tokens=tokens, parent=parent,
                u_accept=u_acc, u_bonus=u_bon)
    eps = max(TIE_TOL, 2.0 * float(err.max()))
    stats = compare_accept(gpu, arrs, orc, tie_tol=eps, bonus_delta=max(BONUS_DELTA, eps))
    print(f"B={B} N={N} V={V}: max|dlogit| {err.max():.3g}, {stats}")
