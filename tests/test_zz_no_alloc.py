"""The allocation-free acceptance entry point, checked against the usual one
and against the oracle.

svf_spec_accept_noalloc is for callers that have no way to give this library
device scratch memory: an inference runtime that hands a plugin only its
input and output buffers, or a serving loop that reserved all device memory
at start-up and may not allocate afterwards. It runs the same kernels as
svf_spec_accept with their scratch in an array the library owns, so it must
return exactly what svf_spec_accept returns on the same inputs -- and keep
doing so on the next call, although that call reuses the same array with
whatever the previous call left in it. Vocabularies above 262144 take the
streaming kernels, which are the ones that use the array; the calls below
run two of those in a row, with different shapes and chunk counts, between
two on-chip calls.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_common import compare_accept

pytestmark = pytest.mark.gpu


def _case(seed, B, N, V):
    rng = np.random.default_rng(seed)
    parent = np.array([-1] + [(i - 1) // 2 for i in range(1, N)], np.int32)
    tgt = (3.0 * rng.standard_normal((B, N, V))).astype(np.float32)
    dft = (tgt + 1.5 * rng.standard_normal((B, N, V))).astype(np.float32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            d = dft[b, parent[c]].astype(np.float64)
            q = np.exp(d - d.max())
            tokens[b, c] = rng.choice(V, p=q / q.sum())
    return dict(target=tgt, draft=dft, tokens=tokens,
                parent=np.broadcast_to(parent, (B, N)).copy(),
                u_accept=rng.random((B, N), dtype=np.float32),
                u_bonus=rng.random(B, dtype=np.float32))


def test_noalloc_accept_matches_workspace_accept_on_two_calls():
    assert torch.cuda.is_available(), "GPU test"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as sv
    lib = sv.load_library()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    # calls in a row with different shapes: each must not see what the one
    # before it left in the array (the two streamed ones use it)
    used = []
    for seed, B, N, V in ((5, 8, 15, 32000), (7, 2, 7, 300000), (8, 3, 15, 524288),
                          (6, 3, 31, 128256)):
        need = sv.spec_accept_workspace_size(B, N, V)
        used.append(need)
        arrs = _case(seed, B, N, V)
        a = {k: torch.from_numpy(v).to(dev) for k, v in arrs.items()}
        ref = sv.spec_accept(a["target"], a["draft"], a["tokens"], a["parent"], a["u_accept"],
                             a["u_bonus"])
        acc_len = torch.full((B,), -7, dtype=torch.int32, device=dev)
        path = torch.full((B, N), -7, dtype=torch.int32, device=dev)
        out_tok = torch.full((B, N), -7, dtype=torch.int32, device=dev)
        ratio = torch.full((B, N), 7.0, dtype=torch.float32, device=dev)
        status = torch.full((B,), -7, dtype=torch.int32, device=dev)
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        rc = lib.svf_spec_accept_noalloc(
            P(a["target"]), P(a["draft"]), P(a["tokens"]), P(a["parent"]), P(a["u_accept"]),
            P(a["u_bonus"]), B, N, V, P(acc_len), P(path), P(out_tok), P(ratio), P(status),
            ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, sv.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(status, ref["status"])
        assert torch.equal(acc_len, ref["accept_len"])
        assert torch.equal(path, ref["path"])
        assert torch.equal(out_tok, ref["out_tokens"])
        np.testing.assert_array_equal(ratio.cpu().numpy(), ref["ratio"].cpu().numpy())
        gpu = {"accept_len": acc_len.cpu().numpy(), "path": path.cpu().numpy(),
               "out_tokens": out_tok.cpu().numpy(), "ratio": ratio.cpu().numpy(),
               "status": status.cpu().numpy()}
        compare_accept(gpu, arrs, oracle.spec_accept(**arrs))
    assert used[1] > 0 and used[2] > 0 and used[1] != used[2], used


def test_noalloc_rejects_requests_beyond_its_scratch():
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as sv
    lib = sv.load_library()
    P = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    B, N, V = 4096, 1024, 786432
    rc = lib.svf_spec_accept_noalloc(P, P, P, P, P, P, B, N, V, P, P, P, None, P, None)
    assert rc == sv.SVF_ERR_SCRATCH_LIMIT
