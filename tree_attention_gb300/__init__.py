"""Python binding of ``libtreeattn.so``, the sm_103a batched tree-attention
library (C ABI in ``include/tree_attn.h``).

The binding only marshals arguments: tensors are passed to the C entry points
as raw device pointers, every step of the computation runs in the library's
CUDA kernels, and there is no CPU fallback.  If the library has not been
built, importing works but every call raises ``RuntimeError``.

The operation is ``batch_tree_attn`` of the page "tree_attn.py"
(python/tvm/relax/frontend/nn/llm/tree_attn.py): ragged, multi-sequence GQA
attention over a causal prefix plus each q row's tree ancestors (DFS
``[enter, exit)`` intervals, ``_check_tree_order``), with optional inline
rotate-half RoPE (``_rope`` of the page "_kernel_common.py"), emitting the
output and the base-2 log-sum-exp.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "TA_OK", "TA_ERR_INVALID_ARGUMENT", "TA_ERR_UNSUPPORTED", "TA_ERR_CUDA",
    "TA_ERR_DEVICE_TIMEOUT", "TreeAttnError", "Dims", "lib", "lib_path", "workspace_size",
    "tree_attn", "plan", "run", "device_status", "status_string", "mask_dense", "check_inputs",
    "TreeAttention", "PagedDims", "make_paged_dims", "paged_workspace_size", "tree_attn_paged",
    "MAX_CHUNKS", "split_workspace_size", "tree_attn_split", "merge_states", "last_cuda_error",
    "folds_rotation", "noalloc_device_status", "set_wait_hooks", "auto_split_chunks",
    "set_scheduler",
]

TA_OK = 0
TA_ERR_INVALID_ARGUMENT = 1
TA_ERR_UNSUPPORTED = 2
TA_ERR_CUDA = 3
TA_ERR_DEVICE_TIMEOUT = 4
TA_FP16 = 0
TA_BF16 = 1
MAX_CHUNKS = 16   # split-KV: most chunks per (sequence, q tile) pair

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libtreeattn.so")


class TreeAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {status_string(status)} ({status})"
        if status == TA_ERR_CUDA:
            msg += f": {last_cuda_error()}"
        super().__init__(msg)
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("total_kv", ctypes.c_int32), ("total_tree", ctypes.c_int32),
                ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("rotary_mode", ctypes.c_int32)]


class PagedDims(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("total_tree", ctypes.c_int32), ("h_q", ctypes.c_int32),
                ("h_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int), ("num_pages", ctypes.c_int32),
                ("nnz_pages", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(lib_path):
        raise RuntimeError(f"libtreeattn.so is not built ({lib_path}); run "
                           "tree_attention_gb300.build.build() or __graft_entry__.build()")
    L = ctypes.CDLL(lib_path)
    vp, i32p, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t
    L.tree_attn_workspace_size.argtypes = [ctypes.POINTER(Dims)]
    L.tree_attn_workspace_size.restype = sz
    L.tree_attn.argtypes = [vp, i32p, vp, vp, i32p, i32p, i32p, i32p, vp, vp, ctypes.c_int32,
                            ctypes.c_float, ctypes.c_float, ctypes.c_float,
                            ctypes.POINTER(Dims), vp, sz, vp]
    L.tree_attn.restype = ctypes.c_int
    L.tree_attn_plan.argtypes = [i32p, i32p, i32p, i32p, i32p, ctypes.c_int32, ctypes.c_float,
                                 ctypes.c_float, ctypes.POINTER(Dims), vp, sz, vp]
    L.tree_attn_plan.restype = ctypes.c_int
    L.tree_attn_run.argtypes = [vp, vp, vp, i32p, i32p, i32p, i32p, i32p, vp, vp,
                                ctypes.c_int32, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                ctypes.POINTER(Dims), vp, sz, vp]
    L.tree_attn_run.restype = ctypes.c_int
    L.tree_attn_noalloc.argtypes = [vp, i32p, vp, vp, i32p, i32p, i32p, i32p, vp, vp,
                                    ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, ctypes.POINTER(Dims), vp]
    L.tree_attn_noalloc.restype = ctypes.c_int
    L.tree_attn_device_status.argtypes = [vp, vp]
    L.tree_attn_device_status.restype = ctypes.c_int
    L.tree_attn_noalloc_device_status.argtypes = [vp]
    L.tree_attn_noalloc_device_status.restype = ctypes.c_int
    L.tree_attn_set_wait_hooks.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    L.tree_attn_set_wait_hooks.restype = ctypes.c_int
    L.tree_attn_last_cuda_error.argtypes = []
    L.tree_attn_last_cuda_error.restype = ctypes.c_char_p
    L.tree_attn_status_string.argtypes = [ctypes.c_int]
    L.tree_attn_status_string.restype = ctypes.c_char_p
    L.tree_attn_mask_dense.argtypes = [i32p, i32p, i32p, i32p, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, vp, vp]
    L.tree_attn_mask_dense.restype = ctypes.c_int
    L.tree_attn_check_inputs.argtypes = [i32p, i32p, i32p, i32p, i32p, ctypes.POINTER(Dims)]
    L.tree_attn_check_inputs.restype = ctypes.c_int
    L.tree_attn_paged_workspace_size.argtypes = [ctypes.POINTER(PagedDims)]
    L.tree_attn_paged_workspace_size.restype = sz
    L.tree_attn_paged.argtypes = [vp, i32p, vp, i32p, i32p, i32p, i32p, i32p, vp, vp,
                                  ctypes.c_int32, ctypes.c_float, ctypes.POINTER(PagedDims), vp,
                                  sz, vp]
    L.tree_attn_paged.restype = ctypes.c_int
    L.tree_attn_split_workspace_size.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32]
    L.tree_attn_split_workspace_size.restype = sz
    L.tree_attn_set_scheduler.argtypes = [ctypes.c_int32]
    L.tree_attn_set_scheduler.restype = ctypes.c_int
    L.tree_attn_auto_split_chunks.argtypes = [ctypes.POINTER(Dims)]
    L.tree_attn_auto_split_chunks.restype = ctypes.c_int32
    L.tree_attn_split.argtypes = [vp, i32p, vp, vp, i32p, i32p, i32p, i32p, vp, vp,
                                  ctypes.c_int32, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Dims), vp, sz,
                                  vp]
    L.tree_attn_split.restype = ctypes.c_int
    L.tree_attn_merge_states.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int, vp, vp, vp]
    L.tree_attn_merge_states.restype = ctypes.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    try:
        return lib().tree_attn_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def last_cuda_error() -> str:
    """The CUDA error behind this thread's most recent TA_ERR_CUDA."""
    try:
        return lib().tree_attn_last_cuda_error().decode()
    except RuntimeError:
        return "unknown"


def folds_rotation(total_kv: int, device=None) -> bool:
    """Whether the one-call entry points fold the key rotation into the plan
    kernel (problems of at most 64 kv tokens per SM), i.e. launch two kernels
    instead of three under RoPE."""
    idx = torch.cuda.current_device() if device is None else device
    return total_kv <= 64 * torch.cuda.get_device_properties(idx).multi_processor_count


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return TA_FP16
    if t == torch.bfloat16:
        return TA_BF16
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_dims(q: torch.Tensor, k: torch.Tensor, q_indptr: torch.Tensor,
              tree_order: torch.Tensor, rotary_mode: int = 0) -> Dims:
    return Dims(batch_size=q_indptr.numel() - 1, total_q=q.shape[0], total_kv=k.shape[0],
                total_tree=tree_order.shape[0], h_q=q.shape[1], h_kv=k.shape[1],
                head_dim=q.shape[2], dtype=_dtype_code(q.dtype), rotary_mode=int(rotary_mode))


def workspace_size(dims: Dims) -> int:
    return int(lib().tree_attn_workspace_size(ctypes.byref(dims)))


def auto_split_chunks(dims: Dims) -> int:
    """The split-KV chunk cap ``tree_attn`` uses for ``dims`` on the current
    device (1: no split; 0: invalid dims)."""
    return int(lib().tree_attn_auto_split_chunks(ctypes.byref(dims)))


def _check_dev(name: str, t: Optional[torch.Tensor], dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def tree_attn(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order, out, lse,
              rotary_mode: int, rope_scale: float, rope_theta: float, sm_scale: float,
              workspace: torch.Tensor, stream=None) -> None:
    """Enqueue one batched tree attention on ``stream`` (default: torch's
    current stream).  All tensors are CUDA tensors with the layouts of
    ``include/tree_attn.h``; ``out`` and ``lse`` are written."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_dev(name, t, q.dtype)
    for name, t in (("q_indptr", q_indptr), ("kv_indptr", kv_indptr), ("mn_indptr", mn_indptr),
                    ("tree_order", tree_order), ("q_rope_position", q_rope_position)):
        _check_dev(name, t, torch.int32)
    _check_dev("lse", lse, torch.float32)
    _check_dev("workspace", workspace)
    dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
    st = lib().tree_attn(_ptr(q), _ptr(q_indptr), _ptr(k), _ptr(v), _ptr(kv_indptr),
                         _ptr(q_rope_position), _ptr(mn_indptr), _ptr(tree_order), _ptr(out),
                         _ptr(lse), int(rotary_mode), float(rope_scale), float(rope_theta),
                         float(sm_scale), ctypes.byref(dims), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn")


def tree_attn_noalloc(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order,
                      out, lse, rotary_mode: int, rope_scale: float, rope_theta: float,
                      sm_scale: float, stream=None) -> None:
    """``tree_attn`` for callers that may not allocate device memory: the
    library's static 32 MiB device scratch array serves as the workspace.
    Calls share that array, so they must not overlap on the GPU."""
    dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
    st = lib().tree_attn_noalloc(_ptr(q), _ptr(q_indptr), _ptr(k), _ptr(v), _ptr(kv_indptr),
                                 _ptr(q_rope_position), _ptr(mn_indptr), _ptr(tree_order),
                                 _ptr(out), _ptr(lse), int(rotary_mode), float(rope_scale),
                                 float(rope_theta), float(sm_scale), ctypes.byref(dims),
                                 _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_noalloc")


def make_paged_dims(q: torch.Tensor, pages: torch.Tensor, q_indptr: torch.Tensor,
                    page_values: torch.Tensor, tree_order: torch.Tensor) -> PagedDims:
    return PagedDims(batch_size=q_indptr.numel() - 1, total_q=q.shape[0],
                     total_tree=tree_order.shape[0], h_q=q.shape[1], h_kv=pages.shape[2],
                     head_dim=q.shape[2], dtype=_dtype_code(q.dtype), num_pages=pages.shape[0],
                     nnz_pages=page_values.numel())


def paged_workspace_size(dims: PagedDims) -> int:
    return int(lib().tree_attn_paged_workspace_size(ctypes.byref(dims)))


def tree_attn_paged(q, q_indptr, pages, page_indptr, page_values, length_info, mn_indptr,
                    tree_order, out, lse, rotary_mode: int, sm_scale: float,
                    workspace: torch.Tensor, stream=None) -> None:
    """Enqueue tree attention over a paged KV cache (``pages [num_pages, 2,
    h_kv, 16, d]``, page table ``page_indptr``/``page_values``, last-page
    lengths ``length_info``); layouts as in ``include/tree_attn.h``."""
    for name, t in (("q", q), ("pages", pages), ("out", out)):
        _check_dev(name, t, q.dtype)
    for name, t in (("q_indptr", q_indptr), ("page_indptr", page_indptr),
                    ("page_values", page_values), ("length_info", length_info),
                    ("mn_indptr", mn_indptr), ("tree_order", tree_order)):
        _check_dev(name, t, torch.int32)
    _check_dev("lse", lse, torch.float32)
    _check_dev("workspace", workspace)
    if pages.dim() != 5 or pages.shape[1] != 2 or pages.shape[3] != 16:
        raise ValueError("pages must be [num_pages, 2, h_kv, 16, head_dim]")
    dims = make_paged_dims(q, pages, q_indptr, page_values, tree_order)
    st = lib().tree_attn_paged(_ptr(q), _ptr(q_indptr), _ptr(pages), _ptr(page_indptr),
                               _ptr(page_values), _ptr(length_info), _ptr(mn_indptr),
                               _ptr(tree_order), _ptr(out), _ptr(lse), int(rotary_mode),
                               float(sm_scale), ctypes.byref(dims), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_paged")


def split_workspace_size(dims: Dims, max_chunks: int) -> int:
    return int(lib().tree_attn_split_workspace_size(ctypes.byref(dims), int(max_chunks)))


def tree_attn_split(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order, out,
                    lse, rotary_mode: int, rope_scale: float, rope_theta: float,
                    sm_scale: float, max_chunks: int, chunk_tiles: int,
                    workspace: torch.Tensor, stream=None) -> None:
    """``tree_attn`` with split-KV: pairs with many kv tiles are cut into up
    to ``max_chunks`` chunks of about ``chunk_tiles`` 128-column tiles (0: the
    plan picks the length), whose partial states a merge kernel combines.
    ``workspace`` holds ``split_workspace_size(dims, max_chunks)`` bytes."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_dev(name, t, q.dtype)
    for name, t in (("q_indptr", q_indptr), ("kv_indptr", kv_indptr), ("mn_indptr", mn_indptr),
                    ("tree_order", tree_order), ("q_rope_position", q_rope_position)):
        _check_dev(name, t, torch.int32)
    _check_dev("lse", lse, torch.float32)
    _check_dev("workspace", workspace)
    dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
    st = lib().tree_attn_split(_ptr(q), _ptr(q_indptr), _ptr(k), _ptr(v), _ptr(kv_indptr),
                               _ptr(q_rope_position), _ptr(mn_indptr), _ptr(tree_order),
                               _ptr(out), _ptr(lse), int(rotary_mode), float(rope_scale),
                               float(rope_theta), float(sm_scale), int(max_chunks),
                               int(chunk_tiles), ctypes.byref(dims), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_split")


def merge_states(parts: torch.Tensor, lses: torch.Tensor, out: Optional[torch.Tensor] = None,
                 lse: Optional[torch.Tensor] = None, stream=None):
    """Merge ``n`` attention states over disjoint kv sets: ``parts [n, ...,
    d]`` (fp16/bf16, normalised) and base-2 ``lses [n, ...]`` (float32) into
    ``out [..., d]`` and ``lse [...]`` (returned)."""
    _check_dev("parts", parts)
    _check_dev("lses", lses, torch.float32)
    if parts.dim() < 2 or tuple(lses.shape) != tuple(parts.shape[:-1]):
        raise ValueError("parts must be [n, ..., d] and lses [n, ...]")
    n, d = parts.shape[0], parts.shape[-1]
    rows = lses[0].numel() if n else 0
    if out is None:
        out = torch.empty(parts.shape[1:], dtype=parts.dtype, device=parts.device)
    if lse is None:
        lse = torch.empty(lses.shape[1:], dtype=torch.float32, device=parts.device)
    _check_dev("out", out, parts.dtype)
    _check_dev("lse", lse, torch.float32)
    st = lib().tree_attn_merge_states(_ptr(parts), _ptr(lses), int(n), int(rows), int(d),
                                      _dtype_code(parts.dtype), _ptr(out), _ptr(lse),
                                      _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_merge_states")
    return out, lse


def plan(q, q_indptr, k, kv_indptr, q_rope_position, mn_indptr, tree_order,
         rotary_mode: int, rope_scale: float, rope_theta: float, workspace: torch.Tensor,
         stream=None) -> None:
    """Enqueue the plan kernel (work items, tile classes, RoPE table); q and
    k are passed only for their shapes and dtype."""
    dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
    st = lib().tree_attn_plan(_ptr(q_indptr), _ptr(kv_indptr), _ptr(q_rope_position),
                              _ptr(mn_indptr), _ptr(tree_order), int(rotary_mode),
                              float(rope_scale), float(rope_theta), ctypes.byref(dims),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_plan")


def run(q, k, v, q_indptr, kv_indptr, q_rope_position, mn_indptr, tree_order, out, lse,
        rotary_mode: int, rope_scale: float, rope_theta: float, sm_scale: float,
        workspace: torch.Tensor, stream=None) -> None:
    """Enqueue the key rotation (RoPE) and the attention kernel on the plan
    held in ``workspace``."""
    dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
    st = lib().tree_attn_run(_ptr(q), _ptr(k), _ptr(v), _ptr(q_indptr), _ptr(kv_indptr),
                             _ptr(q_rope_position), _ptr(mn_indptr), _ptr(tree_order), _ptr(out),
                             _ptr(lse), int(rotary_mode), float(rope_scale), float(rope_theta),
                             float(sm_scale), ctypes.byref(dims), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_run")


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    return int(lib().tree_attn_device_status(_ptr(workspace), _stream_ptr(stream)))


def noalloc_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status that
    ``tree_attn_noalloc`` calls left in the library's static scratch array."""
    return int(lib().tree_attn_noalloc_device_status(_stream_ptr(stream)))


def set_wait_hooks(wait_limit_ns: int = 0, stall: bool = False) -> None:
    """Test hook: the bounded-wait limit of later calls on this thread (0:
    the default) and whether their MMA threads first wait on a barrier that
    nothing arrives on (so that the wait runs out)."""
    st = lib().tree_attn_set_wait_hooks(int(wait_limit_ns), 1 if stall else 0)
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_set_wait_hooks")


def set_scheduler(mode: int) -> None:
    """Work scheduling of later calls' attention kernels on this thread: 0
    the atomic work queue, 1 cluster launch control (default)."""
    st = lib().tree_attn_set_scheduler(int(mode))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_set_scheduler")


def mask_dense(q_indptr, kv_indptr, mn_indptr, tree_order, total_q: int, max_kv: int,
               stream=None) -> torch.Tensor:
    """Dense visibility bytes ``[total_q, max_kv]`` from the device mask code."""
    vis = torch.zeros((max(total_q, 1), max(max_kv, 1)), dtype=torch.uint8,
                      device=q_indptr.device)
    st = lib().tree_attn_mask_dense(_ptr(q_indptr), _ptr(kv_indptr), _ptr(mn_indptr),
                                    _ptr(tree_order), q_indptr.numel() - 1, total_q, max_kv,
                                    _ptr(vis), _stream_ptr(stream))
    if st != TA_OK:
        raise TreeAttnError(st, "tree_attn_mask_dense")
    return vis[:total_q, :max_kv]


def check_inputs(q_indptr, kv_indptr, mn_indptr, tree_order, dims: Dims) -> int:
    """Host-side validation of host (CPU) int32 index arrays."""
    import numpy as np
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.int32)) for a in
            (q_indptr, kv_indptr, mn_indptr, tree_order)]
    ptrs = [a.ctypes.data_as(ctypes.c_void_p) if a.size else None for a in arrs]
    return int(lib().tree_attn_check_inputs(ptrs[0], ptrs[1], ptrs[2], ptrs[3], None,
                                            ctypes.byref(dims)))


class TreeAttention:
    """Owns a workspace sized for one problem shape and runs the call.

    ``inputs`` is a dict of CUDA tensors with keys ``q, q_indptr, k, v,
    kv_indptr, q_rope_position (or None), mn_indptr, tree_order``."""

    def __init__(self, q, k, q_indptr, tree_order, rotary_mode: int, rope_scale: float,
                 rope_theta: float, sm_scale: float):
        self.dims = make_dims(q, k, q_indptr, tree_order, rotary_mode)
        n = workspace_size(self.dims)
        if n == 0:
            raise TreeAttnError(TA_ERR_UNSUPPORTED, "tree_attn_workspace_size")
        # zero-filled once: the library keeps its counters consistent afterwards
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
        self.rotary_mode, self.rope_scale = rotary_mode, rope_scale
        self.rope_theta, self.sm_scale = rope_theta, sm_scale

    def __call__(self, q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order,
                 out=None, lse=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        tree_attn(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order, out,
                  lse, self.rotary_mode, self.rope_scale, self.rope_theta, self.sm_scale,
                  self.workspace, stream)
        return out, lse
