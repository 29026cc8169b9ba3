"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up after its deadline, reports SVF_DEV_TIMEOUT, and the
context keeps working."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_tree_03_gb300 import build as _b
    _b.build()
    import speculative_decoding_tree_03_gb300 as m
    return m


@pytest.mark.parametrize("deadline_s", [0.005, 0.05])
def test_wait_runs_out_and_reports(sv, deadline_s):
    r = sv.selftest_wait_timeout(deadline_s)
    timeout = 16
    assert r["cta_status"] == timeout and r["cluster_status"] == timeout
    for k in ("cta_elapsed_s", "cluster_elapsed_s"):
        us = round(r[k] * 1e6)
        assert round(deadline_s * 1e6) <= us < round(deadline_s * 1e6) + 50000, r
    # the context is still usable: a mask build afterwards matches the oracle
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2]], np.int32)
    anc, depth, status = sv.tree_mask_build(torch.from_numpy(parent).cuda())
    torch.cuda.synchronize()
    o_anc, o_depth, _ = oracle.tree_mask(parent)
    assert (anc.cpu().numpy().view(np.uint64) == o_anc).all()
    assert (depth.cpu().numpy() == o_depth).all() and int(status.sum()) == 0


def test_attention_wait_runs_out_and_the_next_call_is_exact(sv):
    """The tensor-core attention kernels with a 1 ns wait deadline: the first
    wait that is not already complete gives up, the CTA drains its copies and
    tensor-core operations in flight, releases its tensor memory, and every
    sequence reports SVF_DEV_TIMEOUT -- with one chunk per unit, with chunks
    merged in a cluster, and in the persistent kernel (whose pieces are still
    published and merged, flagged). With the default deadline restored, the
    next call on the same inputs matches the oracle (so tensor memory was
    freed: a leaked allocation would stall every later CTA's allocation; and
    the persistent kernel's per-unit counters were left at zero)."""
    from test_gpu_parity import _attn_case, _run_attn, BF16_OUT_TOL, BF16_LSE_TOL
    from synth import binary_tree_parent
    lib = sv.load_library()
    B = 3
    parent = np.broadcast_to(binary_tree_parent(4), (B, 31)).copy()
    c = _attn_case(41, B, 31, parent, [2500, 800, 1700], 32, 8, 128, "bf16", 16)
    try:
        for splits, kernel in ((1, 1), (3, 1), (0, 2)):
            assert lib.svf_debug_set_attn_splits(splits) == 0
            assert lib.svf_debug_set_attn_kernel(kernel) == 0
            assert lib.svf_debug_set_attn_wait_ns(1) == 0
            _, _, status = _run_attn(sv, c, "bf16")
            assert ((status & 16) != 0).all(), status
            assert ((status & ~16) == 0).all(), status
            assert lib.svf_debug_set_attn_wait_ns(0) == 0
            out, lse, status = _run_attn(sv, c, "bf16")
            assert (status == 0).all()
            o_ref, l_ref = oracle.tree_attn(c["q"], c["K"], c["V"], c["lens"], c["parent"])
            assert np.abs(out - o_ref.reshape(out.shape)).max() <= BF16_OUT_TOL
            assert np.abs(lse - l_ref.reshape(lse.shape)).max() <= BF16_LSE_TOL
    finally:
        lib.svf_debug_set_attn_wait_ns(0)
        lib.svf_debug_set_attn_splits(0)
        lib.svf_debug_set_attn_kernel(0)
