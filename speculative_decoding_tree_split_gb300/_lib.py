"""ctypes binding of libtreeattn.so (C ABI declared in include/tree_attn.h).

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity, then their data pointers, the sizes and the current CUDA stream
are handed to the library.  Every step of split tree attention runs in the
library's kernels.  There is no fallback: if the library is missing or a
tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreeattn.so")

# Host-side return codes (include/tree_attn.h).
ERRORS = {
    -1: "null pointer",
    -2: "unsupported or inconsistent sizes",
    -3: "misaligned pointer",
    -4: "workspace missing, too small or misaligned",
    -5: "CUDA error",
    -6: "sizes exceed the library's built-in scratch array",
}
STATUS_BAD_PARENT = 1
STATUS_BAD_PAGE = 2
STATUS_BAD_SEQ_LEN = 3
STATUS_TIMEOUT = 4
STATUS_BAD_PATH = 5
MAX_T = 64

EXPORTED = (
    "tree_mask_build",
    "tree_attn_workspace_size",
    "tree_attn_verify",
    "tree_attn_verify_ctas",
    "tree_attn_workspace_size_ctas",
    "tree_attn_version",
    "tree_attn_prefix_pass",
    "tree_attn_suffix_merge",
    "tree_attn_verify_noalloc",
    "tree_mask_build_batched",
    "tree_attn_verify_batched",
    "tree_attn_verify_paged_tree",
    "tree_greedy_accept",
    "tree_kv_commit",
    "tree_dense_mask_build",
    "tree_attn_verify_dense",
    "tree_attn_plan",
    "tree_attn_verify_tree",
    "tree_accept_commit",
    "tree_attn_set_wait_limit_ns",
    "tree_attn_set_early_prefix_loads",
)


class PlanInfo(ctypes.Structure):
    """tree_attn_plan_info of include/tree_attn.h."""

    _fields_ = [("units", ctypes.c_int), ("row_blocks", ctypes.c_int),
                ("replicas", ctypes.c_int), ("n_ctas", ctypes.c_int),
                ("merge_warps_per_row", ctypes.c_int), ("max_steps", ctypes.c_longlong),
                ("workspace_bytes", ctypes.c_size_t), ("tree_in_prefix", ctypes.c_int),
                ("merge_rows_per_warp", ctypes.c_int)]


class TreeAttnError(RuntimeError):
    """A negative return code from the C ABI."""

    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}: {ERRORS.get(code, 'unknown error')}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtreeattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with speculative_decoding_tree_split_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.tree_mask_build.argtypes = [vp, i32, vp, vp, vp]
    lib.tree_mask_build.restype = i32
    lib.tree_attn_workspace_size.argtypes = [i32] * 7
    lib.tree_attn_workspace_size.restype = sz
    lib.tree_attn_workspace_size_ctas.argtypes = [i32] * 7
    lib.tree_attn_workspace_size_ctas.restype = sz
    verify_args = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                   i32, f32, vp, sz, vp, vp]
    lib.tree_attn_verify.argtypes = verify_args
    lib.tree_attn_verify.restype = i32
    lib.tree_attn_verify_ctas.argtypes = verify_args + [i32]
    lib.tree_attn_verify_ctas.restype = i32
    lib.tree_attn_prefix_pass.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                          i32, f32, vp, sz, i32, vp, vp]
    lib.tree_attn_prefix_pass.restype = i32
    lib.tree_attn_suffix_merge.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                           i32, i32, f32, vp, sz, i32, vp]
    lib.tree_attn_suffix_merge.restype = i32
    lib.tree_attn_verify_noalloc.argtypes = verify_args[:19] + [vp, vp]
    lib.tree_attn_verify_noalloc.restype = i32
    lib.tree_mask_build_batched.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.tree_mask_build_batched.restype = i32
    lib.tree_attn_verify_batched.argtypes = verify_args
    lib.tree_attn_verify_batched.restype = i32
    lib.tree_attn_verify_paged_tree.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, vp, vp, i32, i32,
                                                i32, i32, i32, i32, i32, f32, vp, sz, vp, vp]
    lib.tree_attn_verify_paged_tree.restype = i32
    lib.tree_greedy_accept.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp, vp]
    lib.tree_greedy_accept.restype = i32
    lib.tree_kv_commit.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                   i32, i32, vp, vp]
    lib.tree_kv_commit.restype = i32
    lib.tree_dense_mask_build.argtypes = [vp, i32, vp, i32, i32, i32, vp, vp, vp, vp]
    lib.tree_dense_mask_build.restype = i32
    lib.tree_attn_verify_dense.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, vp, vp, i32, i32,
                                           i32, i32, i32, i32, i32, f32, vp, sz, vp, vp]
    lib.tree_attn_verify_dense.restype = i32
    lib.tree_attn_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                   ctypes.POINTER(PlanInfo)]
    lib.tree_attn_plan.restype = i32
    lib.tree_attn_verify_tree.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, vp, vp, vp,
                                          i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp, vp]
    lib.tree_attn_verify_tree.restype = i32
    lib.tree_accept_commit.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                       vp, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.tree_accept_commit.restype = i32
    lib.tree_attn_version.argtypes = []
    lib.tree_attn_version.restype = i32
    lib.tree_attn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.tree_attn_set_wait_limit_ns.restype = ctypes.c_ulonglong
    lib.tree_attn_set_early_prefix_loads.argtypes = [i32]
    lib.tree_attn_set_early_prefix_loads.restype = i32
    if path == LIB_PATH:
        _lib = lib
    return lib


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtypes, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")


_BITS64 = (torch.int64, getattr(torch, "uint64", torch.int64))


def mask_build(parents: torch.Tensor, mask_out: Optional[torch.Tensor] = None,
               status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Ancestor-or-self bitmask per node of a flattened draft tree.

    parents: int32 [T] on the GPU.  Returns int64 [T] holding the uint64 bits.
    """
    _check(parents, "parents", (torch.int32,), 1)
    T = parents.shape[0]
    if mask_out is None:
        mask_out = torch.empty(T, dtype=torch.int64, device=parents.device)
    _check(mask_out, "mask_out", _BITS64, 1)
    if status is not None:
        _check(status, "status", (torch.int32,))
    rc = load().tree_mask_build(_ptr(parents), T, _ptr(mask_out), _ptr(status),
                                _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_mask_build", rc)
    return mask_out


def mask_build_batched(parents: torch.Tensor, mask_out: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Masks of a batch of trees: parents int32 [n][T] -> int64 [n][T] bits."""
    _check(parents, "parents", (torch.int32,), 2)
    n, T = parents.shape
    if mask_out is None:
        mask_out = torch.empty((n, T), dtype=torch.int64, device=parents.device)
    _check(mask_out, "mask_out", _BITS64, 2)
    if status is not None:
        _check(status, "status", (torch.int32,))
    rc = load().tree_mask_build_batched(_ptr(parents), T, n, _ptr(mask_out), _ptr(status),
                                        _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_mask_build_batched", rc)
    return mask_out


def workspace_size(B: int, Hq: int, Hkv: int, d: int, T: int, max_seq_len: int, page_size: int,
                   n_ctas: int = 0) -> int:
    """Workspace bytes tree_attn_verify needs on the current device."""
    if n_ctas:
        return int(load().tree_attn_workspace_size_ctas(B, Hq, Hkv, d, T, page_size, n_ctas))
    return int(load().tree_attn_workspace_size(B, Hq, Hkv, d, T, max_seq_len, page_size))


def verify(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
           block_table: torch.Tensor, seq_lens: torch.Tensor, tree_k: torch.Tensor,
           tree_v: torch.Tensor, mask: torch.Tensor, *, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           status: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
           stream=None, n_ctas: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split tree attention for one layer (see tree_attn_verify in the header).

    q [B][T][Hq][d] bf16; k_pages/v_pages [num_pages][Hkv][P][d] bf16;
    block_table [B][max_pages] int32; seq_lens [B] int32; tree_k/tree_v
    [B][T][Hkv][d] bf16; mask [T] int64/uint64 bits.  Returns (out, lse).
    """
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 4)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(tree_k, "tree_k", bf, 4)
    _check(tree_v, "tree_v", bf, 4)
    _check(mask, "mask", _BITS64, 1)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, d2 = k_pages.shape
    if (d2 != d or tuple(v_pages.shape) != tuple(k_pages.shape)
            or tuple(tree_k.shape) != (B, T, Hkv, d) or tuple(tree_v.shape) != (B, T, Hkv, d)
            or block_table.shape[0] != B or seq_lens.shape[0] != B or mask.shape[0] != T):
        raise ValueError("inconsistent tensor shapes")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    _check(out, "out", bf, 4)
    _check(lse, "lse", (torch.float32,), 3)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, d, T, 0, P, n_ctas)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", (torch.uint8,))
    if status is not None:
        _check(status, "status", (torch.int32,))
    lib = load()
    args = [_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), _ptr(tree_k), _ptr(tree_v), _ptr(mask), _ptr(out), _ptr(lse),
            B, Hq, Hkv, d, T, P, num_pages, float(softmax_scale), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(status), _stream_handle(stream)]
    if n_ctas:
        rc = lib.tree_attn_verify_ctas(*args, int(n_ctas))
    else:
        rc = lib.tree_attn_verify(*args)
    if rc != 0:
        raise TreeAttnError("tree_attn_verify", rc)
    return out, lse


def verify_batched(q, k_pages, v_pages, block_table, seq_lens, tree_k, tree_v, masks, *,
                   out=None, lse=None, workspace=None, status=None, softmax_scale=None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """tree_attn_verify with one tree per sequence (masks [B][T])."""
    _check(masks, "masks", _BITS64, 2)
    return _verify_generic("tree_attn_verify_batched", q, k_pages, v_pages, block_table,
                           seq_lens, tree_k, tree_v, masks, out, lse, workspace, status,
                           softmax_scale, stream)


def verify_tree(q, k_pages, v_pages, block_table, seq_lens, tree_k, tree_v, parents, *,
                mask_out=None, out=None, lse=None, workspace=None, status=None,
                softmax_scale=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Mask build + split tree attention in one call: parents int32 [T] or
    [B][T]; the masks are built on the device (and written to mask_out if
    given)."""
    bf = (torch.bfloat16,)
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"), (tree_k, "tree_k"),
                 (tree_v, "tree_v")):
        _check(t, n, bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(parents, "parents", (torch.int32,))
    if mask_out is not None:
        _check(mask_out, "mask_out", _BITS64)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    stride = T if parents.dim() == 2 else 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, d, T, 0, P)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = load().tree_attn_verify_tree(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(tree_k), _ptr(tree_v), _ptr(parents), stride, _ptr(mask_out),
        _ptr(out), _ptr(lse), B, Hq, Hkv, d, T, P, num_pages, float(softmax_scale),
        _ptr(workspace), workspace.numel(), _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_attn_verify_tree", rc)
    return out, lse


def verify_paged_tree(q, k_pages, v_pages, block_table, seq_lens, mask, *, out=None, lse=None,
                      workspace=None, status=None, softmax_scale=None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split tree attention with the tree tokens' K/V inside the paged cache at
    positions seq_lens[b] .. seq_lens[b] + T - 1; mask [T] or [B][T]."""
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 4)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(mask, "mask", _BITS64)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    mask_stride = T if mask.dim() == 2 else 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, d, T, 0, P)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = load().tree_attn_verify_paged_tree(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(mask), mask_stride, _ptr(out), _ptr(lse), B, Hq, Hkv, d, T, P,
        num_pages, float(softmax_scale), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_attn_verify_paged_tree", rc)
    return out, lse


def _verify_generic(fn, q, k_pages, v_pages, block_table, seq_lens, tree_k, tree_v, mask, out,
                    lse, workspace, status, softmax_scale, stream):
    bf = (torch.bfloat16,)
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"), (tree_k, "tree_k"),
                 (tree_v, "tree_v")):
        _check(t, n, bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, d, T, 0, P)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = getattr(load(), fn)(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(tree_k), _ptr(tree_v), _ptr(mask), _ptr(out), _ptr(lse), B, Hq, Hkv,
        d, T, P, num_pages, float(softmax_scale), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError(fn, rc)
    return out, lse


def plan(B: int, Hq: int, Hkv: int, d: int, T: int, page_size: int, max_pages_per_seq: int,
         sm_count: int = 0) -> dict:
    """The kernel selector's launch choices for these shapes (host only when
    sm_count > 0)."""
    info = PlanInfo()
    rc = load().tree_attn_plan(B, Hq, Hkv, d, T, page_size, max_pages_per_seq, sm_count,
                               ctypes.byref(info))
    if rc != 0:
        raise TreeAttnError("tree_attn_plan", rc)
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def dense_cols_for(max_keys: int) -> int:
    """Row length of an explicit mask covering max_keys cache positions."""
    return max(16, (int(max_keys) + 15) // 16 * 16)


def dense_mask_build(mask, seq_lens, T: int, dense_cols: int, *, dense_out=None, key_lens=None,
                     status=None, stream=None):
    """Explicit [B][T][dense_cols] mask of the one-pass form (tree tokens in
    the cache after each prefix) and key_lens = seq_lens + T."""
    _check(mask, "mask", _BITS64)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    B = seq_lens.shape[0]
    dev = seq_lens.device
    if dense_out is None:
        dense_out = torch.empty((B, T, dense_cols), dtype=torch.uint8, device=dev)
    if key_lens is None:
        key_lens = torch.empty(B, dtype=torch.int32, device=dev)
    stride = T if mask.dim() == 2 else 0
    rc = load().tree_dense_mask_build(_ptr(mask), stride, _ptr(seq_lens), B, T, dense_cols,
                                      _ptr(dense_out), _ptr(key_lens), _ptr(status),
                                      _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_dense_mask_build", rc)
    return dense_out, key_lens


def verify_dense(q, k_pages, v_pages, block_table, key_lens, dense_mask, *, out=None, lse=None,
                 workspace=None, status=None, softmax_scale=None, stream=None):
    """One-pass tree attention under the explicit mask dense_mask [B][T][cols]."""
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 4)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(key_lens, "key_lens", (torch.int32,), 1)
    _check(dense_mask, "dense_mask", (torch.uint8,), 3)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, d, T, 0, P)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = load().tree_attn_verify_dense(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
        _ptr(key_lens), _ptr(dense_mask), dense_mask.shape[2], _ptr(out), _ptr(lse), B, Hq, Hkv,
        d, T, P, num_pages, float(softmax_scale), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_attn_verify_dense", rc)
    return out, lse


def greedy_accept(mask, draft_tokens, target_tokens, *, accept_len=None, accept_path=None,
                  bonus_token=None, stream=None):
    """Greedy acceptance: mask int64 [T] or [B][T]; draft / target int32 [B][T].
    Returns (accept_len [B], accept_path [B][T], bonus_token [B]), int32."""
    _check(mask, "mask", _BITS64)
    _check(draft_tokens, "draft_tokens", (torch.int32,), 2)
    _check(target_tokens, "target_tokens", (torch.int32,), 2)
    B, T = draft_tokens.shape
    if tuple(target_tokens.shape) != (B, T) or mask.shape[-1] != T:
        raise ValueError("draft_tokens, target_tokens and mask disagree on B or T")
    dev = draft_tokens.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if accept_path is None:
        accept_path = torch.empty((B, T), dtype=torch.int32, device=dev)
    if bonus_token is None:
        bonus_token = torch.empty(B, dtype=torch.int32, device=dev)
    stride = T if mask.dim() == 2 else 0
    rc = load().tree_greedy_accept(_ptr(mask), stride, _ptr(draft_tokens), _ptr(target_tokens),
                                   B, T, _ptr(accept_len), _ptr(accept_path), _ptr(bonus_token),
                                   _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_greedy_accept", rc)
    return accept_len, accept_path, bonus_token


def kv_commit(k_pages, v_pages, block_table, seq_lens, accept_path, accept_len, *,
              tree_k=None, tree_v=None, seq_lens_out=None, status=None, stream=None):
    """Write each sequence's accepted path K/V at positions seq_lens[b] + k
    (in place in k_pages / v_pages).  tree_k / tree_v None: the tree tokens
    are in the cache already.  Returns seq_lens_out (seq_lens + accept_len)."""
    bf = (torch.bfloat16,)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(accept_path, "accept_path", (torch.int32,), 2)
    _check(accept_len, "accept_len", (torch.int32,), 1)
    if tree_k is not None:
        _check(tree_k, "tree_k", bf, 4)
        _check(tree_v, "tree_v", bf, 4)
    num_pages, Hkv, P, d = k_pages.shape
    B, T = accept_path.shape
    if seq_lens_out is None:
        seq_lens_out = torch.empty(B, dtype=torch.int32, device=seq_lens.device)
    rc = load().tree_kv_commit(_ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                               block_table.shape[1], _ptr(seq_lens), _ptr(tree_k), _ptr(tree_v),
                               _ptr(accept_path), _ptr(accept_len), _ptr(seq_lens_out), B, Hkv,
                               d, T, P, num_pages, _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_kv_commit", rc)
    return seq_lens_out


def accept_commit(mask, draft_tokens, target_tokens, k_pages, v_pages, block_table, seq_lens, *,
                  tree_k=None, tree_v=None, accept_len=None, accept_path=None, bonus_token=None,
                  seq_lens_out=None, status=None, stream=None):
    """greedy_accept + kv_commit in one launch.  Returns (accept_len, accept_path,
    bonus_token, seq_lens_out)."""
    _check(mask, "mask", _BITS64)
    _check(draft_tokens, "draft_tokens", (torch.int32,), 2)
    _check(target_tokens, "target_tokens", (torch.int32,), 2)
    bf = (torch.bfloat16,)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    B, T = draft_tokens.shape
    num_pages, Hkv, P, d = k_pages.shape
    dev = draft_tokens.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if accept_path is None:
        accept_path = torch.empty((B, T), dtype=torch.int32, device=dev)
    if bonus_token is None:
        bonus_token = torch.empty(B, dtype=torch.int32, device=dev)
    if seq_lens_out is None:
        seq_lens_out = torch.empty(B, dtype=torch.int32, device=dev)
    stride = T if mask.dim() == 2 else 0
    rc = load().tree_accept_commit(
        _ptr(mask), stride, _ptr(draft_tokens), _ptr(target_tokens), _ptr(k_pages), _ptr(v_pages),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(tree_k), _ptr(tree_v),
        _ptr(accept_len), _ptr(accept_path), _ptr(bonus_token), _ptr(seq_lens_out), B, Hkv, d, T,
        P, num_pages, _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_accept_commit", rc)
    return accept_len, accept_path, bonus_token, seq_lens_out


def prefix_pass(q, k_pages, v_pages, block_table, seq_lens, workspace, *, T=None,
                status=None, softmax_scale=None, stream=None, n_ctas: int = 0) -> None:
    """Prefix pass alone: partial results of every split into `workspace`."""
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 4)
    _check(k_pages, "k_pages", bf, 4)
    _check(v_pages, "v_pages", bf, 4)
    _check(block_table, "block_table", (torch.int32,), 2)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(workspace, "workspace", (torch.uint8,))
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    rc = load().tree_attn_prefix_pass(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), B, Hq, Hkv, d, T, P, num_pages, float(softmax_scale), _ptr(workspace),
        workspace.numel(), int(n_ctas), _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_attn_prefix_pass", rc)


def suffix_merge(q, seq_lens, max_pages_per_seq: int, page_size: int, tree_k, tree_v, mask,
                 workspace, out, lse, *, softmax_scale=None, stream=None,
                 n_ctas: int = 0) -> None:
    """Tree-masked suffix pass and log-sum-exp merge of the prefix partials."""
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 4)
    _check(seq_lens, "seq_lens", (torch.int32,), 1)
    _check(tree_k, "tree_k", bf, 4)
    _check(tree_v, "tree_v", bf, 4)
    _check(mask, "mask", _BITS64, 1)
    _check(out, "out", bf, 4)
    _check(lse, "lse", (torch.float32,), 3)
    _check(workspace, "workspace", (torch.uint8,))
    B, T, Hq, d = q.shape
    Hkv = tree_k.shape[2]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    rc = load().tree_attn_suffix_merge(
        _ptr(q), _ptr(seq_lens), int(max_pages_per_seq), _ptr(tree_k), _ptr(tree_v), _ptr(mask),
        _ptr(out), _ptr(lse), B, Hq, Hkv, d, T, int(page_size), float(softmax_scale),
        _ptr(workspace), workspace.numel(), int(n_ctas), _stream_handle(stream))
    if rc != 0:
        raise TreeAttnError("tree_attn_suffix_merge", rc)


DEFAULT_WAIT_NS = 2_000_000_000


def set_wait_limit_ns(ns: int) -> int:
    """Limit (ns) of the prefix pass's internal pipeline waits for calls
    enqueued from now on; 0 restores the default (2 s).  Returns the previous
    limit.  A call whose wait runs out stores STATUS_TIMEOUT in its status."""
    return int(load().tree_attn_set_wait_limit_ns(int(ns)))


def set_early_prefix_loads(enable: bool) -> bool:
    """Promise, for calls enqueued from now on, that the kernel before each
    call in its stream writes none of seq_lens, block_table and the committed
    prefix K/V: the prefix pass then plans and loads its first K/V blocks
    before waiting for that kernel.  Returns the previous setting."""
    return bool(load().tree_attn_set_early_prefix_loads(1 if enable else 0))


def version() -> int:
    return int(load().tree_attn_version())
