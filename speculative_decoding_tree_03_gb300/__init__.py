"""GB300-native one-pass tree verification for EAGLE-style speculative decoding.

A thin ctypes binding over ``libspecverify.so``, whose C ABI is declared in
``include/specverify.h``. The functions here only check tensor shapes, dtypes,
devices and contiguity and pass raw device pointers and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU path: calling with a tensor that is not on a CUDA device, or
without the built library, raises.

    anc, depth, status = tree_mask_build(parent)
    out, lse, status   = tree_verify_attn(q, k_cache, v_cache, page_table, seq_lens, anc)
    res                = spec_accept(target_logits, draft_logits, tokens, parent,
                                     u_accept, u_bonus)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libspecverify.so")

SVF_F32, SVF_BF16 = 0, 1
SVF_OK, SVF_ERR_ARG, SVF_ERR_UNSUPPORTED, SVF_ERR_LAUNCH, SVF_ERR_WORKSPACE = 0, -1, -2, -3, -4
SVF_ERR_SCRATCH_LIMIT = -5
SVF_DEV_BAD_PARENT, SVF_DEV_BAD_TOKEN, SVF_DEV_BAD_PAGE, SVF_DEV_BAD_LENGTH, SVF_DEV_TIMEOUT = (
    1, 2, 4, 8, 16)

EXPORTED = [
    "svf_tree_mask_build",
    "svf_tree_verify_attn_workspace_size",
    "svf_tree_verify_attn",
    "svf_tree_mask_attn",
    "svf_spec_accept_workspace_size",
    "svf_spec_accept",
    "svf_spec_accept_noalloc",
    "svf_lm_head",
    "svf_debug_set_attn_wait_ns",
    "svf_debug_set_attn_splits",
    "svf_debug_set_attn_kernel",
    "svf_spec_accept_lmhead",
    "svf_kv_commit",
    "svf_selftest_wait_timeout",
    "svf_spec_accept_bf16",
    "svf_spec_accept_greedy",
    "svf_spec_accept_onehot",
    "svf_spec_accept_greedy_bf16",
    "svf_spec_accept_onehot_bf16",
    "svf_eagle2_init",
    "svf_eagle2_expand",
    "svf_eagle2_finalize",
    "svf_status_string",
    "svf_version",
]

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecverify.so and declare its signatures (no GPU needed)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise SpecVerifyError(
            f"{path} is missing: build it with speculative_decoding_tree_03_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.svf_tree_mask_build.argtypes = [P, I, I, P, P, P, P]
    lib.svf_tree_mask_build.restype = I
    lib.svf_tree_verify_attn_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.svf_tree_verify_attn_workspace_size.restype = Z
    lib.svf_tree_verify_attn.argtypes = [P, P, P, I, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P,
                                         Z, P, P]
    lib.svf_tree_verify_attn.restype = I
    lib.svf_tree_mask_attn.argtypes = [P, P, P, P, P, P, P, I, I, P, I, P, I, I, I, I, I, I, F,
                                       P, P, P, Z, P, P]
    lib.svf_tree_mask_attn.restype = I
    lib.svf_spec_accept_workspace_size.argtypes = [I, I, I]
    lib.svf_spec_accept_workspace_size.restype = Z
    lib.svf_spec_accept.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P, Z, P, P]
    lib.svf_spec_accept.restype = I
    lib.svf_spec_accept_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.svf_spec_accept_noalloc.restype = I
    lib.svf_spec_accept_bf16.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.svf_spec_accept_bf16.restype = I
    lib.svf_spec_accept_greedy.argtypes = [P, P, P, I, I, I, P, P, P, P, P]
    lib.svf_spec_accept_greedy.restype = I
    lib.svf_spec_accept_onehot.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.svf_spec_accept_onehot.restype = I
    lib.svf_spec_accept_greedy_bf16.argtypes = [P, P, P, I, I, I, P, P, P, P, P]
    lib.svf_spec_accept_greedy_bf16.restype = I
    lib.svf_spec_accept_onehot_bf16.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.svf_spec_accept_onehot_bf16.restype = I
    lib.svf_eagle2_init.argtypes = [P, I, I, P, P, P, P, P, P]
    lib.svf_eagle2_init.restype = I
    lib.svf_eagle2_expand.argtypes = [P, I, I, I, I, P, I, P, P, P, P, P, P, P, P]
    lib.svf_eagle2_expand.restype = I
    lib.svf_eagle2_finalize.argtypes = [I, I, P, P, P, P, P, I, P, P, P, P, P, P]
    lib.svf_eagle2_finalize.restype = I
    lib.svf_selftest_wait_timeout.argtypes = [P, ctypes.c_longlong, P]
    lib.svf_selftest_wait_timeout.restype = I
    lib.svf_kv_commit.argtypes = [P, P, I, ctypes.c_longlong, I, I, P, I, P, P, P, I, I, I, I,
                                  I, P, P, I, P, P, P]
    lib.svf_kv_commit.restype = I
    lib.svf_lm_head.argtypes = [P, P, I, I, I, P, P, P]
    lib.svf_lm_head.restype = I
    lib.svf_spec_accept_lmhead.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, P, P, P, P, P, P,
                                           P]
    lib.svf_spec_accept_lmhead.restype = I
    lib.svf_debug_set_attn_wait_ns.argtypes = [ctypes.c_longlong]
    lib.svf_debug_set_attn_wait_ns.restype = I
    lib.svf_debug_set_attn_splits.argtypes = [I]
    lib.svf_debug_set_attn_splits.restype = I
    lib.svf_debug_set_attn_kernel.argtypes = [I]
    lib.svf_debug_set_attn_kernel.restype = I
    lib.svf_status_string.argtypes = [I]
    lib.svf_status_string.restype = ctypes.c_char_p
    lib.svf_version.argtypes = []
    lib.svf_version.restype = I
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().svf_status_string(int(code)).decode()


def _check(rc: int, what: str) -> None:
    if rc != SVF_OK:
        raise SpecVerifyError(f"{what}: {status_string(rc)} ({rc})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise SpecVerifyError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise SpecVerifyError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise SpecVerifyError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise SpecVerifyError(f"{name} must be contiguous")
    return t


_ZEROED_WS = {}


def _zeroed_workspace(need: int, dev: torch.device) -> torch.Tensor:
    """The attention workspace used when the caller passes none: zero-filled
    once and kept per device (every call leaves it zero-filled). Calls that
    may overlap on the GPU should pass workspaces of their own."""
    key = (dev.type, dev.index if dev.index is not None else torch.cuda.current_device())
    ws = _ZEROED_WS.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros((need,), dtype=torch.uint8, device=dev)
        _ZEROED_WS[key] = ws
    return ws


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return SVF_F32
    if dt == torch.bfloat16:
        return SVF_BF16
    raise SpecVerifyError(f"unsupported dtype {dt}")


# ---------------------------------------------------------------------------
# tree_mask_build
# ---------------------------------------------------------------------------

def tree_mask_build(parent: torch.Tensor, anc: Optional[torch.Tensor] = None,
                    depth: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                    stream=None):
    """Ancestor bitmasks of BFS-flattened trees: parent [B, N] int32 ->
    (anc [B, N, ceil(N/64)] int64 bit patterns, depth [B, N] int32, status [B] int32)."""
    lib = load_library()
    _dev(parent, "parent", torch.int32)
    B, N = parent.shape
    W = max(1, (N + 63) // 64)
    dev = parent.device
    if anc is None:
        anc = torch.empty((B, N, W), dtype=torch.int64, device=dev)
    if depth is None:
        depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(anc, "anc", torch.int64, (B, N, W))
    _dev(depth, "depth", torch.int32, (B, N))
    _dev(status, "status", torch.int32, (B,))
    rc = lib.svf_tree_mask_build(_ptr(parent), B, N, _ptr(anc), _ptr(depth), _ptr(status),
                                 _stream(stream))
    _check(rc, "svf_tree_mask_build")
    return anc, depth, status


# ---------------------------------------------------------------------------
# tree_verify_attn
# ---------------------------------------------------------------------------

def tree_verify_attn_workspace_size(B, N, Hq, Hkv, D, dtype, max_pages, page_size) -> int:
    return int(load_library().svf_tree_verify_attn_workspace_size(
        B, N, Hq, Hkv, D, _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype),
        max_pages, page_size))


def tree_verify_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     page_table: torch.Tensor, seq_lens: torch.Tensor, anc: torch.Tensor,
                     sm_scale: float = 0.0, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, want_lse: bool = True, stream=None):
    """Tree attention against a paged KV cache.

    q [B, N, Hq, D]; k_cache, v_cache [num_pages, page_size, Hkv, D] (same dtype,
    float32 or bfloat16); page_table [B, max_pages] int32; seq_lens [B] int32
    (prefix length, tree excluded); anc [B, N, 1] int64 from tree_mask_build.
    Returns (out [B, N, Hq, D], lse [B, N, Hq] float32 or None, status [B] int32).
    """
    lib = load_library()
    _dev(q, "q")
    B, N, Hq, D = q.shape
    dt = q.dtype
    _dev(k_cache, "k_cache", dt)
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise SpecVerifyError("k_cache head_dim differs from q")
    _dev(v_cache, "v_cache", dt, k_cache.shape)
    _dev(page_table, "page_table", torch.int32)
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise SpecVerifyError("page_table must be [B, max_pages]")
    max_pages = page_table.shape[1]
    _dev(seq_lens, "seq_lens", torch.int32, (B,))
    _dev(anc, "anc", torch.int64)
    if anc.shape[0] != B or anc.shape[1] != N:
        raise SpecVerifyError("anc must be [B, N, W]")
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", dt, q.shape)
    if lse is None and want_lse:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _dev(lse, "lse", torch.float32, (B, N, Hq))
    if status is None:
        status = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(status, "status", torch.int32, (B,))
    code = _dtype_code(dt)
    need = int(lib.svf_tree_verify_attn_workspace_size(B, N, Hq, Hkv, D, code, max_pages,
                                                       page_size))
    if workspace is None and need > 0:
        workspace = _zeroed_workspace(need, dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.svf_tree_verify_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages, page_size, _ptr(page_table), max_pages,
        _ptr(seq_lens), _ptr(anc), B, N, Hq, Hkv, D, code, float(sm_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check(rc, "svf_tree_verify_attn")
    return out, lse, status


def tree_mask_attn(parent: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                   sm_scale: float = 0.0, anc: Optional[torch.Tensor] = None,
                   depth: Optional[torch.Tensor] = None,
                   mask_status: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, want_lse: bool = True, stream=None):
    """tree_mask_build and tree_verify_attn in one call (one kernel for
    bfloat16). Returns (out, lse, status, anc, depth, mask_status)."""
    lib = load_library()
    _dev(q, "q")
    B, N, Hq, D = q.shape
    dt = q.dtype
    _dev(parent, "parent", torch.int32, (B, N))
    _dev(k_cache, "k_cache", dt)
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise SpecVerifyError("k_cache head_dim differs from q")
    _dev(v_cache, "v_cache", dt, k_cache.shape)
    _dev(page_table, "page_table", torch.int32)
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise SpecVerifyError("page_table must be [B, max_pages]")
    max_pages = page_table.shape[1]
    _dev(seq_lens, "seq_lens", torch.int32, (B,))
    dev = q.device
    if anc is None:
        anc = torch.empty((B, N, 1), dtype=torch.int64, device=dev)
    _dev(anc, "anc", torch.int64, (B, N, 1))
    if depth is None:
        depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    _dev(depth, "depth", torch.int32, (B, N))
    if mask_status is None:
        mask_status = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(mask_status, "mask_status", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", dt, q.shape)
    if lse is None and want_lse:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _dev(lse, "lse", torch.float32, (B, N, Hq))
    if status is None:
        status = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(status, "status", torch.int32, (B,))
    code = _dtype_code(dt)
    need = int(lib.svf_tree_verify_attn_workspace_size(B, N, Hq, Hkv, D, code, max_pages,
                                                       page_size))
    if workspace is None and need > 0:
        workspace = _zeroed_workspace(need, dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.svf_tree_mask_attn(
        _ptr(parent), _ptr(anc), _ptr(depth), _ptr(mask_status), _ptr(q), _ptr(k_cache),
        _ptr(v_cache), num_pages, page_size, _ptr(page_table), max_pages, _ptr(seq_lens), B, N,
        Hq, Hkv, D, code, float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        _ptr(status), _stream(stream))
    _check(rc, "svf_tree_mask_attn")
    return out, lse, status, anc, depth, mask_status


# ---------------------------------------------------------------------------
# spec_accept
# ---------------------------------------------------------------------------

def spec_accept_workspace_size(B, N, V) -> int:
    return int(load_library().svf_spec_accept_workspace_size(B, N, V))


def spec_accept(target_logits: torch.Tensor, draft_logits: torch.Tensor, tokens: torch.Tensor,
                parent: torch.Tensor, u_accept: torch.Tensor, u_bonus: torch.Tensor,
                want_ratio: bool = True, workspace: Optional[torch.Tensor] = None,
                outputs: Optional[dict] = None, stream=None) -> dict:
    """Acceptance walk. Returns a dict of device tensors: accept_len [B], path [B, N],
    out_tokens [B, N], ratio [B, N] (or None), status [B]. Logits are float32 or
    bfloat16 (both the same dtype)."""
    lib = load_library()
    _dev(target_logits, "target_logits")
    if target_logits.dtype not in (torch.float32, torch.bfloat16):
        raise SpecVerifyError("logits must be float32 or bfloat16")
    B, N, V = target_logits.shape
    _dev(draft_logits, "draft_logits", target_logits.dtype, (B, N, V))
    _dev(tokens, "tokens", torch.int32, (B, N))
    _dev(parent, "parent", torch.int32, (B, N))
    _dev(u_accept, "u_accept", torch.float32, (B, N))
    _dev(u_bonus, "u_bonus", torch.float32, (B,))
    dev = target_logits.device
    o = outputs if outputs is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["path"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["out_tokens"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["ratio"] = torch.empty((B, N), dtype=torch.float32, device=dev) if want_ratio else None
        o["status"] = torch.empty((B,), dtype=torch.int32, device=dev)
    if target_logits.dtype == torch.bfloat16:
        rc = lib.svf_spec_accept_bf16(
            _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parent), _ptr(u_accept),
            _ptr(u_bonus), B, N, V, _ptr(o["accept_len"]), _ptr(o["path"]),
            _ptr(o["out_tokens"]), _ptr(o.get("ratio")), _ptr(o["status"]), _stream(stream))
        _check(rc, "svf_spec_accept_bf16")
        return o
    need = int(lib.svf_spec_accept_workspace_size(B, N, V))
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib.svf_spec_accept(
        _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parent), _ptr(u_accept),
        _ptr(u_bonus), B, N, V, _ptr(o["accept_len"]), _ptr(o["path"]), _ptr(o["out_tokens"]),
        _ptr(o.get("ratio")), _ptr(workspace), ws_bytes, _ptr(o["status"]), _stream(stream))
    _check(rc, "svf_spec_accept")
    return o


def _variant_outputs(o, B, N, dev, want_ratio):
    if "accept_len" not in o:
        o["accept_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["path"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["out_tokens"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["ratio"] = torch.empty((B, N), dtype=torch.float32, device=dev) if want_ratio else None
        o["status"] = torch.empty((B,), dtype=torch.int32, device=dev)
    return o


def spec_accept_greedy(target_logits: torch.Tensor, tokens: torch.Tensor, parent: torch.Tensor,
                       outputs: Optional[dict] = None, stream=None) -> dict:
    """Temperature-0 acceptance (argmax matching) on float32 or bfloat16
    logits. Returns a dict of device tensors: accept_len [B], path [B, N],
    out_tokens [B, N], status [B]."""
    lib = load_library()
    if target_logits.dtype not in (torch.float32, torch.bfloat16):
        raise SpecVerifyError("target_logits must be float32 or bfloat16")
    _dev(target_logits, "target_logits")
    bf = target_logits.dtype == torch.bfloat16
    B, N, V = target_logits.shape
    _dev(tokens, "tokens", torch.int32, (B, N))
    _dev(parent, "parent", torch.int32, (B, N))
    o = _variant_outputs(outputs if outputs is not None else {}, B, N, target_logits.device,
                         False)
    fn = lib.svf_spec_accept_greedy_bf16 if bf else lib.svf_spec_accept_greedy
    rc = fn(_ptr(target_logits), _ptr(tokens), _ptr(parent), B, N, V, _ptr(o["accept_len"]),
            _ptr(o["path"]), _ptr(o["out_tokens"]), _ptr(o["status"]), _stream(stream))
    _check(rc, "svf_spec_accept_greedy" + ("_bf16" if bf else ""))
    return o


def spec_accept_onehot(target_logits: torch.Tensor, tokens: torch.Tensor, parent: torch.Tensor,
                       u_accept: torch.Tensor, u_bonus: torch.Tensor, want_ratio: bool = True,
                       outputs: Optional[dict] = None, stream=None) -> dict:
    """The sampling rule with q = one-hot(candidate) for every child, on
    float32 or bfloat16 logits. Returns accept_len, path, out_tokens, ratio
    (or None) and status."""
    lib = load_library()
    if target_logits.dtype not in (torch.float32, torch.bfloat16):
        raise SpecVerifyError("target_logits must be float32 or bfloat16")
    _dev(target_logits, "target_logits")
    bf = target_logits.dtype == torch.bfloat16
    B, N, V = target_logits.shape
    _dev(tokens, "tokens", torch.int32, (B, N))
    _dev(parent, "parent", torch.int32, (B, N))
    _dev(u_accept, "u_accept", torch.float32, (B, N))
    _dev(u_bonus, "u_bonus", torch.float32, (B,))
    o = _variant_outputs(outputs if outputs is not None else {}, B, N, target_logits.device,
                         want_ratio)
    fn = lib.svf_spec_accept_onehot_bf16 if bf else lib.svf_spec_accept_onehot
    rc = fn(_ptr(target_logits), _ptr(tokens), _ptr(parent), _ptr(u_accept), _ptr(u_bonus), B,
            N, V, _ptr(o["accept_len"]), _ptr(o["path"]), _ptr(o["out_tokens"]),
            _ptr(o.get("ratio")), _ptr(o["status"]), _stream(stream))
    _check(rc, "svf_spec_accept_onehot" + ("_bf16" if bf else ""))
    return o


# ---------------------------------------------------------------------------
# LM head (target logits from hidden states) and the walk fed by it
# ---------------------------------------------------------------------------

def lm_head(hidden: torch.Tensor, weight: torch.Tensor, logits: Optional[torch.Tensor] = None,
            status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """logits[..., v] = hidden[..., :] . weight[v, :] for bf16 hidden [..., H]
    and weight [V, H], as fp32 [..., V]."""
    lib = load_library()
    _dev(hidden, "hidden", torch.bfloat16)
    H = hidden.shape[-1]
    _dev(weight, "weight", torch.bfloat16)
    if weight.dim() != 2 or weight.shape[1] != H:
        raise SpecVerifyError("weight must be [V, H] with H = hidden.shape[-1]")
    V = weight.shape[0]
    R = hidden.numel() // H if H > 0 else 0
    shape = tuple(hidden.shape[:-1]) + (V,)
    if logits is None:
        logits = torch.empty(shape, dtype=torch.float32, device=hidden.device)
    _dev(logits, "logits", torch.float32, shape)
    if status is not None:
        _dev(status, "status", torch.int32)
    rc = lib.svf_lm_head(_ptr(hidden), _ptr(weight), R, H, V, _ptr(logits), _ptr(status),
                         _stream(stream))
    _check(rc, "svf_lm_head")
    return logits


def spec_accept_lmhead(hidden: torch.Tensor, weight: torch.Tensor, draft_logits: torch.Tensor,
                       tokens: torch.Tensor, parent: torch.Tensor, u_accept: torch.Tensor,
                       u_bonus: torch.Tensor, want_ratio: bool = True,
                       outputs: Optional[dict] = None, stream=None) -> dict:
    """The acceptance walk with target rows from the LM head: hidden [B, N, H]
    bf16, weight [V, H] bf16, draft logits [B, N, V] fp32. Returns
    spec_accept's outputs plus "target_logits" [B, N, V] fp32 and
    "lm_status" [1]."""
    lib = load_library()
    _dev(hidden, "hidden", torch.bfloat16)
    B, N, H = hidden.shape
    _dev(weight, "weight", torch.bfloat16)
    V = weight.shape[0]
    if weight.dim() != 2 or weight.shape[1] != H:
        raise SpecVerifyError("weight must be [V, H] with H = hidden.shape[-1]")
    _dev(draft_logits, "draft_logits", torch.float32, (B, N, V))
    _dev(tokens, "tokens", torch.int32, (B, N))
    _dev(parent, "parent", torch.int32, (B, N))
    _dev(u_accept, "u_accept", torch.float32, (B, N))
    _dev(u_bonus, "u_bonus", torch.float32, (B,))
    dev = hidden.device
    o = outputs if outputs is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["path"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["out_tokens"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["ratio"] = torch.empty((B, N), dtype=torch.float32, device=dev) if want_ratio else None
        o["status"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["target_logits"] = torch.empty((B, N, V), dtype=torch.float32, device=dev)
        o["lm_status"] = torch.zeros((1,), dtype=torch.int32, device=dev)
    rc = lib.svf_spec_accept_lmhead(
        _ptr(hidden), _ptr(weight), _ptr(draft_logits), _ptr(tokens), _ptr(parent),
        _ptr(u_accept), _ptr(u_bonus), B, N, H, V, _ptr(o["target_logits"]),
        _ptr(o["accept_len"]), _ptr(o["path"]), _ptr(o["out_tokens"]), _ptr(o.get("ratio")),
        _ptr(o["lm_status"]), _ptr(o["status"]), _stream(stream))
    _check(rc, "svf_spec_accept_lmhead")
    return o


# ---------------------------------------------------------------------------
# EAGLE-2 tree construction
# ---------------------------------------------------------------------------

def eagle2_init(pool: dict, root_tokens: torch.Tensor, stream=None) -> dict:
    """Reset ``pool`` to the roots alone (a new build in the same arrays)."""
    lib = load_library()
    _dev(root_tokens, "root_tokens", torch.int32)
    B, C = pool["parent"].shape
    if root_tokens.shape != (B,):
        raise SpecVerifyError("root_tokens must be [B]")
    rc = lib.svf_eagle2_init(_ptr(root_tokens), B, C, _ptr(pool["parent"]),
                             _ptr(pool["depth"]), _ptr(pool["token"]), _ptr(pool["value"]),
                             _ptr(pool["count"]), _stream(stream))
    _check(rc, "svf_eagle2_init")
    return pool


def eagle2_pool(root_tokens: torch.Tensor, capacity: int, stream=None) -> dict:
    """A node pool per sequence holding only the root (device tensors)."""
    _dev(root_tokens, "root_tokens", torch.int32)
    B = root_tokens.shape[0]
    dev = root_tokens.device
    pool = {"parent": torch.empty((B, capacity), dtype=torch.int32, device=dev),
            "depth": torch.empty((B, capacity), dtype=torch.int32, device=dev),
            "token": torch.empty((B, capacity), dtype=torch.int32, device=dev),
            "value": torch.empty((B, capacity), dtype=torch.float64, device=dev),
            "count": torch.empty((B,), dtype=torch.int32, device=dev)}
    return eagle2_init(pool, root_tokens, stream)


def eagle2_expand(pool: dict, draft_rows: torch.Tensor, frontier: torch.Tensor, k: int,
                  next_frontier: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One expansion round in place; returns the next frontier [B, k].
    ``status`` [B] int32, when given, gets 0 or SVF_DEV_TIMEOUT per sequence."""
    lib = load_library()
    _dev(draft_rows, "draft_rows", torch.float32)
    B, R, V = draft_rows.shape
    _dev(frontier, "frontier", torch.int32, (B, R))
    C = pool["parent"].shape[1]
    if next_frontier is None:
        next_frontier = torch.empty((B, k), dtype=torch.int32, device=draft_rows.device)
    if status is not None:
        _dev(status, "status", torch.int32, (B,))
    rc = lib.svf_eagle2_expand(_ptr(draft_rows), B, R, V, k, _ptr(frontier), C,
                               _ptr(pool["parent"]), _ptr(pool["depth"]), _ptr(pool["token"]),
                               _ptr(pool["value"]), _ptr(pool["count"]), _ptr(next_frontier),
                               None if status is None else _ptr(status), _stream(stream))
    _check(rc, "svf_eagle2_expand")
    return next_frontier


def eagle2_finalize(pool: dict, n_nodes: int, outputs: Optional[dict] = None,
                    stream=None) -> dict:
    """Rerank and flatten: parent [B, n], tokens, values, cids, n_out."""
    lib = load_library()
    B, C = pool["parent"].shape
    dev = pool["parent"].device
    out = outputs if outputs is not None else {}
    if "parent" not in out:
        out.update({"parent": torch.empty((B, n_nodes), dtype=torch.int32, device=dev),
                    "tokens": torch.empty((B, n_nodes), dtype=torch.int32, device=dev),
                    "values": torch.empty((B, n_nodes), dtype=torch.float64, device=dev),
                    "cids": torch.empty((B, n_nodes), dtype=torch.int32, device=dev),
                    "n_out": torch.empty((B,), dtype=torch.int32, device=dev)})
    rc = lib.svf_eagle2_finalize(B, C, _ptr(pool["parent"]), _ptr(pool["depth"]),
                                 _ptr(pool["token"]), _ptr(pool["value"]), _ptr(pool["count"]),
                                 n_nodes, _ptr(out["parent"]), _ptr(out["tokens"]),
                                 _ptr(out["values"]), _ptr(out["cids"]), _ptr(out["n_out"]),
                                 _stream(stream))
    _check(rc, "svf_eagle2_finalize")
    return out


def selftest_wait_timeout(deadline_s: float = 0.02, device="cuda", stream=None) -> dict:
    """Run the bounded-wait diagnostic; returns the statuses and elapsed
    times (seconds) of a CTA wait and a cluster wait that nothing completes."""
    lib = load_library()
    res = torch.zeros((4,), dtype=torch.int32, device=device)
    rc = lib.svf_selftest_wait_timeout(_ptr(res), int(deadline_s * 1e9), _stream(stream))
    _check(rc, "svf_selftest_wait_timeout")
    r = res.cpu().tolist()
    return {"cta_status": r[0], "cta_elapsed_s": r[1] * 1e-6,
            "cluster_status": r[2], "cluster_elapsed_s": r[3] * 1e-6}


# ---------------------------------------------------------------------------
# kv_commit
# ---------------------------------------------------------------------------

def kv_commit(k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
              seq_lens: torch.Tensor, path: torch.Tensor, accept_len: torch.Tensor,
              max_free: Optional[int] = None, outputs: Optional[dict] = None,
              stream=None) -> dict:
    """Keep the accepted path's K/V in place, in path order after the prefix.

    k_cache, v_cache [layers, num_pages, page_size, Hkv, D] (or without the
    layer axis), float32 or bfloat16, each layer contiguous; page_table
    [B, max_pages], seq_lens [B], path [B, N], accept_len [B] int32. Returns a
    dict of device tensors: new_seq_lens [B], freed [B, max_free] (page ids, -1
    padded), n_freed [B], status [B]."""
    lib = load_library()
    _dev(k_cache, "k_cache")
    if k_cache.dim() == 4:
        layers, (num_pages, page_size, Hkv, D) = 1, k_cache.shape
        stride = 0
    elif k_cache.dim() == 5:
        layers, num_pages, page_size, Hkv, D = k_cache.shape
        stride = k_cache.stride(0)
    else:
        raise SpecVerifyError("k_cache must be [layers,] num_pages, page_size, Hkv, D")
    if not (k_cache[0] if k_cache.dim() == 5 else k_cache).is_contiguous():
        raise SpecVerifyError("each layer of k_cache must be contiguous")
    _dev(v_cache, "v_cache", k_cache.dtype, k_cache.shape)
    if v_cache.stride() != k_cache.stride():
        raise SpecVerifyError("v_cache must have k_cache's strides")
    _dev(page_table, "page_table", torch.int32)
    B, max_pages = page_table.shape
    _dev(seq_lens, "seq_lens", torch.int32, (B,))
    _dev(path, "path", torch.int32)
    if path.dim() != 2 or path.shape[0] != B:
        raise SpecVerifyError("path must be [B, N]")
    N = path.shape[1]
    _dev(accept_len, "accept_len", torch.int32, (B,))
    if max_free is None:
        max_free = (N + page_size - 1) // page_size
    dev = k_cache.device
    o = outputs if outputs is not None else {}
    if "status" not in o:
        o["new_seq_lens"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["freed"] = torch.empty((B, max(max_free, 1)), dtype=torch.int32, device=dev)
        o["n_freed"] = torch.empty((B,), dtype=torch.int32, device=dev)
        o["status"] = torch.empty((B,), dtype=torch.int32, device=dev)
    rc = lib.svf_kv_commit(
        _ptr(k_cache), _ptr(v_cache), layers, stride, num_pages, page_size, _ptr(page_table),
        max_pages, _ptr(seq_lens), _ptr(path), _ptr(accept_len), B, N, Hkv, D,
        _dtype_code(k_cache.dtype), _ptr(o["new_seq_lens"]), _ptr(o["freed"]), max_free,
        _ptr(o["n_freed"]), _ptr(o["status"]), _stream(stream))
    _check(rc, "svf_kv_commit")
    return o


# ---------------------------------------------------------------------------
# One verify step: mask -> attention -> acceptance
# ---------------------------------------------------------------------------

def verify_step(parent, tokens, q, k_cache, v_cache, page_table, seq_lens, target_logits,
                draft_logits, u_accept, u_bonus, stream=None, buffers: Optional[dict] = None):
    """The whole hot path on device tensors: ancestor masks and tree attention
    of one layer (one fused call), then the acceptance walk. ``buffers``
    (optional) holds preallocated outputs and workspaces and is filled on the
    first call."""
    bufs = buffers if buffers is not None else {}
    if "attn_ws" not in bufs:
        B, N, Hq, D = q.shape
        need = tree_verify_attn_workspace_size(B, N, Hq, k_cache.shape[2], D, q.dtype,
                                               page_table.shape[1], k_cache.shape[1])
        bufs["attn_ws"] = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    out, lse, astatus, anc, depth, mstatus = tree_mask_attn(
        parent, q, k_cache, v_cache, page_table, seq_lens, anc=bufs.get("anc"),
        depth=bufs.get("depth"), mask_status=bufs.get("mask_status"), out=bufs.get("attn_out"),
        lse=bufs.get("lse"), workspace=bufs["attn_ws"], status=bufs.get("attn_status"),
        stream=stream)
    bufs["anc"], bufs["depth"], bufs["mask_status"] = anc, depth, mstatus
    bufs["attn_out"], bufs["lse"], bufs["attn_status"] = out, lse, astatus
    if "acc_ws" not in bufs:
        B, N, V = target_logits.shape
        bufs["acc_ws"] = torch.empty((spec_accept_workspace_size(B, N, V),), dtype=torch.uint8,
                                     device=q.device)
    res = spec_accept(target_logits, draft_logits, tokens, parent, u_accept, u_bonus,
                      workspace=bufs["acc_ws"], outputs=bufs.get("accept"), stream=stream)
    bufs["accept"] = res
    return out, lse, res, bufs
