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
