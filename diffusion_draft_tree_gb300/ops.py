"""Python binding of libddtree.so (include/ddtree.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks dtypes/shapes/devices,
passes raw device pointers and the current CUDA stream to the C ABI, and turns
a non-OK status into an exception.  All arithmetic runs in the library's CUDA
kernels; there is no CPU path.  If the library has not been built, importing
this module raises instead of falling back.

Names and argument order follow the C ABI: ddtree_topk, ddtree_build,
ddtree_tree_attn, ddtree_accept (one DDTree round, "Accelerating Speculative
Decoding with Block Diffusion Draft Trees" §3-§4.3), plus helpers that allocate
the outputs with torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libddtree.so")

BF16, FP32 = 0, 1
OP_TOPK, OP_TREE_ATTN, OP_ACCEPT = 0, 2, 3
MAX_K, MAX_L, MAX_N = 32, 16, 1024

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error",
          4: "kernel recorded bad device data or a timeout"}


class DDTreeError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: int = 0):
        msg = f"{fn}: {STATUS.get(status, status)}"
        if status == 3:
            msg += f" ({lib.ddtree_last_cuda_error().decode()})"
        if detail:
            msg += f" (detail 0x{detail:08x})"
        super().__init__(msg)
        self.status = status
        self.detail = detail


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                 ctypes.c_float, ctypes.c_size_t)
    lib.ddtree_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i64]
    lib.ddtree_workspace_size.restype = sz
    lib.ddtree_topk.argtypes = [P, i32, i32, i32, i64, i32, P, P, P, P, sz, P]
    lib.ddtree_build.argtypes = [P, P, P, P, i32, i32, i32, i32] + [P] * 9 + [P]
    lib.ddtree_build_heap.argtypes = lib.ddtree_build.argtypes
    lib.ddtree_tree_attn.argtypes = [P, P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                     P, P, P, sz, P]
    lib.ddtree_accept.argtypes = [P, i32, i64, P, P, P, i32, i32, i32, i32, f32, u64, u64, P, P,
                                  P, P, P, P, sz, P]
    lib.ddtree_commit.argtypes = [P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32, P]
    lib.ddtree_accept_path.argtypes = [P, i32, i64, P, P, P, i32, i32, i32, i32, f32, u64, u64,
                                       P, P, P, P, P, P]
    lib.ddtree_topk_noalloc.argtypes = [P, i32, i32, i32, i64, i32, P, P, P, P]
    lib.ddtree_device_check.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.ddtree_selftest_wait.argtypes = [ctypes.c_uint32, P]
    lib.ddtree_last_cuda_error.argtypes = []
    lib.ddtree_last_cuda_error.restype = ctypes.c_char_p
    lib.ddtree_status_str.argtypes = [i32]
    lib.ddtree_status_str.restype = ctypes.c_char_p
    for f in ("ddtree_topk", "ddtree_build", "ddtree_build_heap", "ddtree_tree_attn",
              "ddtree_accept", "ddtree_accept_path", "ddtree_commit", "ddtree_topk_noalloc",
              "ddtree_device_check", "ddtree_selftest_wait"):
        getattr(lib, f).restype = i32
    return lib


lib = _load()

EXPORTED = ("ddtree_workspace_size", "ddtree_topk", "ddtree_build", "ddtree_build_heap",
            "ddtree_tree_attn", "ddtree_accept", "ddtree_device_check", "ddtree_last_cuda_error",
            "ddtree_status_str")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("ddtree kernels take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("ddtree kernels take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise DDTreeError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


def workspace_size(op: int, B=0, L=0, N=0, V=0, K=0, dtype=BF16, Hq=0, Hkv=0, D=0,
                   cache_cap=0) -> int:
    return int(lib.ddtree_workspace_size(op, B, L, N, V, K, dtype, Hq, Hkv, D, cache_cap))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace (torch allocations are)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------
# raw calls (caller-provided outputs), same names as the C ABI
# --------------------------------------------------------------------------

def ddtree_topk(draft_logits, K, topk_idx, topk_logp, lse=None, workspace=None, stream=None):
    """draft_logits [rows][V] (bf16/fp32) -> topk_idx int32 [rows][K], topk_logp fp32."""
    rows, V = draft_logits.shape[0], draft_logits.shape[-1]
    ws = workspace
    _check("ddtree_topk", lib.ddtree_topk(
        _ptr(draft_logits), _dtype_code(draft_logits), rows, V, V, K, _ptr(topk_idx),
        _ptr(topk_logp), _ptr(lse), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))


def ddtree_build(topk_logp, topk_idx, bonus, prefix_len, N, out: dict, stream=None,
                 heap=False):
    """heap=False: the level-synchronous build; heap=True: ddtree_build_heap."""
    B, L, K = topk_logp.shape
    fn = lib.ddtree_build_heap if heap else lib.ddtree_build
    _check("ddtree_build", fn(
        _ptr(topk_logp), _ptr(topk_idx), _ptr(bonus), _ptr(prefix_len), B, L, K, N,
        _ptr(out["parent"]), _ptr(out["depth"]), _ptr(out["rank"]), _ptr(out["token"]),
        _ptr(out["pos_id"]), _ptr(out["score"]), _ptr(out["child_count"]),
        _ptr(out["anc_mask"]), _ptr(out["n_nodes"]), _stream(stream)))


def ddtree_tree_attn(q, k_cache, v_cache, k_tree, v_tree, prefix_len, n_nodes, anc_mask, out,
                     lse=None, scale=None, workspace=None, stream=None):
    B, R, Hq, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    scale = float(scale) if scale is not None else D ** -0.5
    ws = workspace
    _check("ddtree_tree_attn", lib.ddtree_tree_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), cap, _ptr(k_tree), _ptr(v_tree), _ptr(prefix_len),
        _ptr(n_nodes), _ptr(anc_mask), B, R - 1, Hq, Hkv, D, scale, _ptr(out), _ptr(lse),
        _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def ddtree_accept(target_logits, parent, token, n_nodes, L, out: dict, temperature=0.0, seed=0,
                  step=0, workspace=None, stream=None):
    B, R, V = target_logits.shape
    ws = workspace
    _check("ddtree_accept", lib.ddtree_accept(
        _ptr(target_logits), _dtype_code(target_logits), V, _ptr(parent), _ptr(token),
        _ptr(n_nodes), B, L, R - 1, V, float(temperature), int(seed), int(step),
        _ptr(out.get("target_token")), _ptr(out["accept_len"]), _ptr(out["accepted_nodes"]),
        _ptr(out["out_tokens"]), _ptr(out["next_bonus"]), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)))


def ddtree_accept_path(target_logits, parent, token, n_nodes, L, out: dict, temperature=0.0,
                       seed=0, step=0, stream=None):
    """The walk reading only the rows on the accepted path (same outputs as
    ddtree_accept; target_token on the path only)."""
    B, R, V = target_logits.shape
    _check("ddtree_accept_path", lib.ddtree_accept_path(
        _ptr(target_logits), _dtype_code(target_logits), V, _ptr(parent), _ptr(token),
        _ptr(n_nodes), B, L, R - 1, V, float(temperature), int(seed), int(step),
        _ptr(out.get("target_token")), _ptr(out["accept_len"]), _ptr(out["accepted_nodes"]),
        _ptr(out["out_tokens"]), _ptr(out["next_bonus"]), _stream(stream)))


def accept_path(target_logits, tree: dict, L: int, temperature=0.0, seed=0, step=0,
                stream=None) -> dict:
    B, R, V = target_logits.shape
    out = accept_buffers(B, L, R - 1, target_logits.device)
    ddtree_accept_path(target_logits, tree["parent"], tree["token"], tree["n_nodes"], L, out,
                       temperature, seed, step, stream)
    return out


def ddtree_commit(k_cache, v_cache, k_tree, v_tree, accept_len, accepted_nodes, prefix_len,
                  stream=None):
    """Commit the accepted path (root + accepted nodes) to the KV cache in place
    and advance prefix_len in place."""
    B, Hkv, cap, D = k_cache.shape
    R = k_tree.shape[1]
    L = accepted_nodes.shape[1]
    _check("ddtree_commit", lib.ddtree_commit(
        _ptr(k_cache), _ptr(v_cache), cap, _ptr(k_tree), _ptr(v_tree), _ptr(accept_len),
        _ptr(accepted_nodes), _ptr(prefix_len), B, L, R - 1, Hkv, D, _stream(stream)))


def ddtree_selftest_wait(limit_us: int, stream=None):
    """Enqueues a bounded wait that runs out (see include/ddtree.h)."""
    _check("ddtree_selftest_wait", lib.ddtree_selftest_wait(int(limit_us), _stream(stream)))


def ddtree_device_check(stream=None) -> int:
    """Synchronises the stream; raises DDTreeError if a kernel recorded an error."""
    detail = ctypes.c_uint32(0)
    st = lib.ddtree_device_check(_stream(stream), ctypes.byref(detail))
    if st != 0:
        raise DDTreeError("ddtree_device_check", st, detail.value)
    return 0


# --------------------------------------------------------------------------
# allocating helpers
# --------------------------------------------------------------------------

def topk(draft_logits: torch.Tensor, K: int, workspace=None, stream=None):
    """[..., V] logits -> (idx int32 [..., K], logp fp32 [..., K], lse fp32 [...])."""
    lead = draft_logits.shape[:-1]
    x = draft_logits.reshape(-1, draft_logits.shape[-1])
    dev = x.device
    idx = torch.empty((x.shape[0], K), dtype=torch.int32, device=dev)
    lp = torch.empty((x.shape[0], K), dtype=torch.float32, device=dev)
    lse = torch.empty((x.shape[0],), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(OP_TOPK, B=x.shape[0], L=1, V=x.shape[1],
                                                   K=K, dtype=_dtype_code(x)), dev)
    ddtree_topk(x, K, idx, lp, lse, workspace, stream)
    return idx.reshape(*lead, K), lp.reshape(*lead, K), lse.reshape(lead)


def tree_buffers(B: int, N: int, device) -> dict:
    R, W = N + 1, (N + 1 + 31) // 32
    t = {k: torch.empty((B, R), dtype=torch.int32, device=device)
         for k in ("parent", "depth", "rank", "token", "pos_id", "child_count")}
    t["score"] = torch.empty((B, R), dtype=torch.float32, device=device)
    t["anc_mask"] = torch.empty((B, R, W), dtype=torch.int32, device=device)
    t["n_nodes"] = torch.empty((B,), dtype=torch.int32, device=device)
    return t


def build(topk_logp, topk_idx, bonus, prefix_len, N: int, stream=None, heap=False) -> dict:
    B = topk_logp.shape[0]
    t = tree_buffers(B, N, topk_logp.device)
    ddtree_build(topk_logp, topk_idx, bonus, prefix_len, N, t, stream, heap)
    return t


def tree_attn(q, k_cache, v_cache, k_tree, v_tree, prefix_len, n_nodes, anc_mask, scale=None,
              want_lse=True, workspace=None, stream=None):
    B, R, Hq, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, R, Hq), dtype=torch.float32, device=q.device) if want_lse else None
    if workspace is None:
        workspace = alloc_workspace(workspace_size(OP_TREE_ATTN, B=B, N=R - 1, Hq=Hq,
                                                   Hkv=k_cache.shape[1], D=D,
                                                   cache_cap=k_cache.shape[2]), q.device)
    ddtree_tree_attn(q, k_cache, v_cache, k_tree, v_tree, prefix_len, n_nodes, anc_mask, out, lse,
                     scale, workspace, stream)
    return out, lse


def accept_buffers(B: int, L: int, N: int, device) -> dict:
    return {"target_token": torch.empty((B, N + 1), dtype=torch.int32, device=device),
            "accept_len": torch.empty((B,), dtype=torch.int32, device=device),
            "accepted_nodes": torch.empty((B, L), dtype=torch.int32, device=device),
            "out_tokens": torch.empty((B, L + 1), dtype=torch.int32, device=device),
            "next_bonus": torch.empty((B,), dtype=torch.int32, device=device)}


def accept(target_logits, tree: dict, L: int, temperature=0.0, seed=0, step=0, workspace=None,
           stream=None) -> dict:
    B, R, V = target_logits.shape
    out = accept_buffers(B, L, R - 1, target_logits.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(OP_ACCEPT, B=B, N=R - 1, V=V,
                                                   dtype=_dtype_code(target_logits)),
                                    target_logits.device)
    ddtree_accept(target_logits, tree["parent"], tree["token"], tree["n_nodes"], L, out,
                  temperature, seed, step, workspace, stream)
    return out
