"""The C-ABI library builds, loads without a GPU and exports every symbol
include/specverify.h declares; host-side argument checks return their codes
before any CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_tree_03_gb300 import build as b
    b.build()
    import speculative_decoding_tree_03_gb300 as sv
    return sv.load_library()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "specverify.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*\*?\s*(svf_\w+)\s*\(",
                                 text, re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("svf_tree_mask_build", "svf_tree_verify_attn", "svf_spec_accept",
              "svf_tree_verify_attn_workspace_size", "svf_spec_accept_workspace_size",
              "svf_status_string", "svf_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import speculative_decoding_tree_03_gb300 as sv
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert sorted(sv.EXPORTED) == declared_symbols()


def test_status_strings(lib):
    import speculative_decoding_tree_03_gb300 as sv
    assert sv.status_string(0) == "ok"
    assert "workspace" in sv.status_string(-4)
    assert "parent" in sv.status_string(1)
    assert lib.svf_version() >= 100


P = ctypes.c_void_p(256)  # never dereferenced: every call below returns before using it


def test_mask_argument_checks(lib):
    assert lib.svf_tree_mask_build(P, -1, 4, P, P, P, None) == -1
    assert lib.svf_tree_mask_build(None, 0, 4, None, None, None, None) == 0
    assert lib.svf_tree_mask_build(P, 1, 1025, P, P, P, None) == -2
    assert lib.svf_tree_mask_build(P, 1, 0, P, P, P, None) == -2
    assert lib.svf_tree_mask_build(None, 1, 4, P, P, P, None) == -1


def _attn(lib, **kw):
    a = dict(q=P, k=P, v=P, num_pages=4, page_size=16, table=P, max_pages=2, lens=P, anc=P, B=1,
             N=3, Hq=8, Hkv=2, D=128, dtype=1, scale=0.0, out=P, lse=None, ws=None, wsb=0,
             status=P)
    a.update(kw)
    return lib.svf_tree_verify_attn(a["q"], a["k"], a["v"], a["num_pages"], a["page_size"],
                                    a["table"], a["max_pages"], a["lens"], a["anc"], a["B"],
                                    a["N"], a["Hq"], a["Hkv"], a["D"], a["dtype"], a["scale"],
                                    a["out"], a["lse"], a["ws"], a["wsb"], a["status"], None)


def test_attention_argument_checks(lib):
    assert _attn(lib, B=-1) == -1
    assert _attn(lib, B=0, q=None) == 0
    assert _attn(lib, q=None) == -1
    assert _attn(lib, N=65) == -2
    assert _attn(lib, Hq=6, Hkv=4) == -2
    assert _attn(lib, D=64) == -2                       # bf16 needs head_dim 128
    assert _attn(lib, page_size=48) == -2               # bf16 page sizes 16/32/64/128k
    assert _attn(lib, dtype=0, D=96) == -2              # fp32 head_dim 64 or 128
    assert _attn(lib, dtype=7) == -2
    assert _attn(lib, q=ctypes.c_void_p(264)) == -1     # not 16-byte aligned


def test_accept_argument_checks(lib):
    def call(B=2, N=3, V=100, ws=P, wsb=1 << 20, t=P):
        return lib.svf_spec_accept(t, P, P, P, P, P, B, N, V, P, P, P, None, ws, wsb, P, None)
    assert call(B=-1) == -1
    assert call(B=0, t=None) == 0
    assert call(t=None) == -1
    assert call(N=0) == -2 and call(N=1025) == -2
    assert call(V=786433) == -2
    # vocabularies held on chip need no workspace; larger ones stream from
    # memory with a statistics pre-pass that does
    assert lib.svf_spec_accept_workspace_size(2, 3, 100) == 0
    assert lib.svf_spec_accept_workspace_size(64, 31, 262144) == 0
    assert lib.svf_spec_accept_workspace_size(2, 3, 262145) > 0
    assert call(V=300000, ws=None) == -4
    assert call(V=300000, wsb=8) == -4


def test_kv_commit_argument_checks(lib):
    def call(B=2, N=7, layers=1, stride=0, num_pages=8, ps=4, max_pages=4, Hkv=2, D=64,
             dtype=1, max_free=2, freed=P, k=P):
        return lib.svf_kv_commit(k, P, layers, stride, num_pages, ps, P, max_pages, P, P, P, B, N,
                                 Hkv, D, dtype, P, freed, max_free, None, P, None)
    assert call(B=-1) == -1
    assert call(B=0, k=None) == 0
    assert call(k=None) == -1
    assert call(max_free=2, freed=None) == -1          # freed_pages needed when max_free > 0
    assert call(N=0) == -2 and call(N=1025) == -2
    assert call(dtype=5) == -2
    assert call(Hkv=1, D=4) == -2                       # a row of 8 bytes is not 16-byte sized
    assert call(layers=2, stride=100) == -1             # layers overlap
    assert call(k=ctypes.c_void_p(264)) == -1           # not 16-byte aligned


def test_accept_bf16_argument_checks(lib):
    def call(B=2, N=3, V=100, t=P):
        return lib.svf_spec_accept_bf16(t, P, P, P, P, P, B, N, V, P, P, P, None, P, None)
    assert call(B=-1) == -1
    assert call(B=0, t=None) == 0
    assert call(t=None) == -1
    assert call(N=0) == -2 and call(N=1025) == -2
    assert call(V=262145) == -2                      # only on-chip vocabularies
    assert call(t=ctypes.c_void_p(260)) == -1        # 8-byte loads of four bf16


def test_accept_variant_argument_checks(lib):
    def greedy(B=2, N=3, V=100, t=P):
        return lib.svf_spec_accept_greedy(t, P, P, B, N, V, P, P, P, P, None)

    def onehot(B=2, N=3, V=100, t=P, u=P):
        return lib.svf_spec_accept_onehot(t, P, P, u, P, B, N, V, P, P, P, None, P, None)
    for call in (greedy, onehot):
        assert call(B=-1) == -1
        assert call(B=0, t=None) == 0
        assert call(t=None) == -1
        assert call(N=0) == -2 and call(N=1025) == -2
        assert call(V=786433) == -2                        # beyond the streamed vocabularies
        assert call(V=128, t=ctypes.c_void_p(260)) == -1   # float4 loads need 16-byte rows
    assert onehot(u=None) == -1


def test_accept_variant_bf16_argument_checks(lib):
    def greedy(B=2, N=3, V=100, t=P):
        return lib.svf_spec_accept_greedy_bf16(t, P, P, B, N, V, P, P, P, P, None)

    def onehot(B=2, N=3, V=100, t=P, u=P):
        return lib.svf_spec_accept_onehot_bf16(t, P, P, u, P, B, N, V, P, P, P, None, P, None)
    for call in (greedy, onehot):
        assert call(B=-1) == -1
        assert call(B=0, t=None) == 0
        assert call(t=None) == -1
        assert call(N=0) == -2 and call(N=1025) == -2
        assert call(V=786433) == -2                        # beyond the streamed vocabularies
        assert call(V=128, t=ctypes.c_void_p(260)) == -1   # 8-byte loads of four bf16
    assert onehot(u=None) == -1


def test_eagle2_argument_checks(lib):
    def expand(B=2, R=8, V=1000, k=8, cap=329, rows=P):
        return lib.svf_eagle2_expand(rows, B, R, V, k, P, cap, P, P, P, P, P, P, None, None)
    assert expand(B=-1) == -1
    assert expand(B=0, rows=None) == 0
    assert expand(rows=None) == -1
    assert expand(k=0) == -2 and expand(k=17) == -2
    assert expand(V=4, k=8) == -2                    # k > V
    assert expand(V=(1 << 20) + 1) == -2             # beyond the draft vocabulary bound
    assert expand(cap=2049) == -2
    assert expand(R=65536) == -2


def test_selftest_argument_checks(lib):
    assert lib.svf_selftest_wait_timeout(None, 10 ** 6, None) == -1
    assert lib.svf_selftest_wait_timeout(P, 10, None) == -1          # below 1 us
    assert lib.svf_selftest_wait_timeout(P, 2 * 10 ** 9, None) == -1  # above 1 s


def test_workspace_sizes_without_gpu(lib):
    # bf16 with Hq / Hkv a power of two: the persistent kernel's pieces (two
    # slots per SM of 256 fp32 rows of 128, their log-sum-exps and flags)
    # and then two counters per unit, each part rounded up to 256 bytes
    up = lambda x: (x + 255) // 256 * 256
    sms = 148  # the library's stand-in without a device
    def expect(B, N, Hq, Hkv):
        M = N * (Hq // Hkv)
        rows = 256 if M > 128 else 128
        units = B * Hkv * -(-M // rows)
        return (up(2 * sms * 32 * 256 * 16) + up(2 * sms * 256 * 4) + up(2 * sms * 4)
                + up(units * 8))
    assert lib.svf_tree_verify_attn_workspace_size(1, 31, 32, 8, 128, 1, 1, 2176) == expect(1, 31, 32, 8)
    assert lib.svf_tree_verify_attn_workspace_size(64, 31, 64, 8, 128, 1, 2051, 16) == \
        expect(64, 31, 64, 8)
    assert lib.svf_tree_verify_attn_workspace_size(16, 64, 64, 8, 128, 1, 256, 16) == \
        expect(16, 64, 64, 8)
    # fp32 and a non-power-of-two group size need none
    assert lib.svf_tree_verify_attn_workspace_size(1, 31, 32, 8, 128, 0, 1, 2176) == 0
    assert lib.svf_tree_verify_attn_workspace_size(1, 31, 24, 8, 128, 1, 1, 2176) == 0
    # the hook that picks the bf16 kernel checks its argument
    assert lib.svf_debug_set_attn_kernel(3) == -1
    assert lib.svf_debug_set_attn_kernel(-1) == -1
    assert lib.svf_debug_set_attn_kernel(0) == 0


def test_package_refuses_cpu_tensors():
    import torch
    import speculative_decoding_tree_03_gb300 as sv
    with pytest.raises(sv.SpecVerifyError):
        sv.tree_mask_build(torch.zeros((1, 3), dtype=torch.int32))


def test_package_checks_before_any_launch():
    """Every binding call validates its tensors on the host: CPU tensors, a
    wrong logits dtype and a wrong status shape raise before the library is
    asked to launch anything."""
    import torch
    import speculative_decoding_tree_03_gb300 as sv
    t = torch.zeros((1, 3, 16), dtype=torch.float32)
    i = torch.zeros((1, 3), dtype=torch.int32)
    u = torch.zeros((1, 3), dtype=torch.float32)
    ub = torch.zeros((1,), dtype=torch.float32)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_accept_greedy(t, i, i)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_accept_onehot(t, i, i, u, ub)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_accept_greedy(t.to(torch.float16), i, i)          # neither fp32 nor bf16
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_accept(t, t, i, i, u, ub)
    with pytest.raises(sv.SpecVerifyError):
        sv.eagle2_pool(torch.zeros((2,), dtype=torch.int32), 16)


def test_lm_head_argument_checks(lib):
    import speculative_decoding_tree_03_gb300 as sv
    P = ctypes.c_void_p(256)
    Q = ctypes.c_void_p(257)  # not 16-byte aligned
    assert lib.svf_lm_head(None, P, 4, 64, 10, P, None, None) == sv.SVF_ERR_ARG
    assert lib.svf_lm_head(P, P, 4, 100, 10, P, None, None) == sv.SVF_ERR_UNSUPPORTED
    assert lib.svf_lm_head(P, P, 4, 64, 0, P, None, None) == sv.SVF_ERR_UNSUPPORTED
    assert lib.svf_lm_head(Q, P, 4, 64, 10, P, None, None) == sv.SVF_ERR_ARG
    assert lib.svf_lm_head(P, P, 0, 64, 10, P, None, None) == sv.SVF_OK
    assert lib.svf_lm_head(P, P, -1, 64, 10, P, None, None) == sv.SVF_ERR_ARG
    args = [P] * 7 + [2, 3, 64, 300000] + [P] * 4 + [None, None, P, None]
    assert lib.svf_spec_accept_lmhead(*args) == sv.SVF_ERR_UNSUPPORTED   # V beyond on-chip
    args = [P] * 7 + [2, 3, 64, 1000] + [P] * 4 + [None, None, None, None]
    assert lib.svf_spec_accept_lmhead(*args) == sv.SVF_ERR_ARG           # no status


def test_debug_hooks(lib):
    import speculative_decoding_tree_03_gb300 as sv
    assert lib.svf_debug_set_attn_splits(9) == sv.SVF_ERR_ARG
    assert lib.svf_debug_set_attn_splits(-1) == sv.SVF_ERR_ARG
    assert lib.svf_debug_set_attn_splits(0) == sv.SVF_OK
    assert lib.svf_debug_set_attn_wait_ns(0) == sv.SVF_OK


def test_fused_mask_attention_argument_checks(lib):
    import speculative_decoding_tree_03_gb300 as sv
    P = ctypes.c_void_p(256)
    # parent missing
    args = [None, P, P, P, P, P, P, 10, 16, P, 4, P, 2, 7, 8, 2, 128, 1, 0.0, P, P, None, 0, P,
            None]
    assert lib.svf_tree_mask_attn(*args) == sv.SVF_ERR_ARG
    # N above the attention limit
    args = [P, P, P, P, P, P, P, 10, 16, P, 4, P, 2, 65, 8, 2, 128, 1, 0.0, P, P, None, 0, P,
            None]
    assert lib.svf_tree_mask_attn(*args) == sv.SVF_ERR_UNSUPPORTED
    # fp32 needs the mask outputs (that path reads the masks from memory)
    args = [P, None, None, None, P, P, P, 10, 16, P, 4, P, 2, 7, 8, 2, 128, 0, 0.0, P, P, None,
            0, P, None]
    assert lib.svf_tree_mask_attn(*args) == sv.SVF_ERR_ARG
