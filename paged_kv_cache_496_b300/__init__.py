"""Python binding of libpagedkv.so, the B300 (sm_103a) paged KV-cache hot path.

Argument marshalling only: every step of the path runs in the library's CUDA kernels. torch is
used for device memory and streams. The functions mirror the C ABI in include/pagedkv.h:

    kv_store(k, v, slot_mapping, k_cache, v_cache)
    paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=...)
    paged_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, block_tables, scale, k_cache, v_cache)

Caches are [num_blocks, block_size, num_kv_heads, head_dim] bf16 (the layout of the PagedAttention
pages: fixed-size blocks addressed through per-sequence block tables). There is no CPU fallback:
importing this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = ["kv_store", "decode_plan", "paged_decode", "paged_prefill", "get_device_error",
           "PagedKVError", "lib", "CacheDesc", "DecodePlan", "LIBRARY"]

LIBRARY = _build.LIBRARY

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE_TOO_SMALL = -3
PKV_ERR_CUDA = -4

DEVERR_BAD_SLOT = 1
DEVERR_BAD_BLOCK = 2
DEVERR_CTX_CLAMPED = 4
DEVERR_TIMEOUT = 8
DEVERR_BAD_LENGTHS = 16
DEVERR_INTERNAL = 32

DECODE_ENGINE_CUDA_CORE = 1    # PKV_DECODE_ENGINE_CUDA_CORE
DECODE_ENGINE_TENSOR_CORE = 2  # PKV_DECODE_ENGINE_TENSOR_CORE
DECODE_PLAN_REUSE = 1          # PKV_DECODE_PLAN_REUSE


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("split_tokens", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("auto_split", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("engine", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


ABI_VERSION = 202  # PKV_VERSION of include/pagedkv.h that the argtypes below describe


def _load():
    if not os.path.exists(LIBRARY):
        raise ImportError(f"{LIBRARY} is missing: build it with `python "
                          "paged_kv_cache_496_b300/build.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIBRARY)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    L.pkv_kv_store.restype = ctypes.c_int
    L.pkv_kv_store.argtypes = [vp, vp, vp, i32, vp, vp, CacheDesc, vp]
    L.pkv_decode_plan_make.restype = ctypes.c_int
    L.pkv_decode_plan_make.argtypes = [i32, i32, CacheDesc, i32, i32, ctypes.POINTER(DecodePlan)]
    L.pkv_paged_decode.restype = ctypes.c_int
    L.pkv_paged_decode.argtypes = [vp, vp, vp, CacheDesc, vp, i32, vp, i32, i32, f32,
                                   ctypes.POINTER(DecodePlan), vp, vp, sz, vp]
    L.pkv_paged_decode_store.restype = ctypes.c_int
    L.pkv_paged_decode_store.argtypes = [vp, vp, vp, vp, vp, vp, CacheDesc, vp, i32, vp, i32,
                                         i32, f32, ctypes.POINTER(DecodePlan), vp, vp, sz, vp]
    L.pkv_prefill_workspace_bytes.restype = ctypes.c_size_t
    L.pkv_prefill_workspace_bytes.argtypes = [i32]
    L.pkv_paged_prefill.restype = ctypes.c_int
    L.pkv_paged_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, vp, vp,
                                    CacheDesc, i32, f32, vp, vp, sz, vp]
    L.pkv_copy_blocks.restype = ctypes.c_int
    L.pkv_copy_blocks.argtypes = [vp, vp, CacheDesc, vp, i32, vp]
    L.pkv_gather_blocks.restype = ctypes.c_int
    L.pkv_gather_blocks.argtypes = [vp, vp, CacheDesc, vp, i32, vp, vp, vp]
    L.pkv_scatter_blocks.restype = ctypes.c_int
    L.pkv_scatter_blocks.argtypes = [vp, vp, vp, i32, vp, vp, CacheDesc, vp]
    L.pkv_block_hashes.restype = ctypes.c_int
    L.pkv_block_hashes.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    L.pkv_selftest_bounded_wait.restype = ctypes.c_int
    L.pkv_selftest_bounded_wait.argtypes = [vp]
    L.pkv_get_device_error.restype = ctypes.c_int
    L.pkv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_last_error.restype = ctypes.c_char_p
    L.pkv_last_error.argtypes = []
    L.pkv_version.restype = ctypes.c_int
    L.pkv_version.argtypes = []
    if L.pkv_version() != ABI_VERSION:
        raise ImportError(f"{LIBRARY} has ABI version {L.pkv_version()}, this binding declares "
                          f"{ABI_VERSION}: rebuild it with `python paged_kv_cache_496_b300/build.py`")
    return L


lib = _load()


def _check(status: int):
    if status != PKV_OK:
        msg = lib.pkv_last_error().decode() or lib.pkv_status_string(status).decode()
        raise PagedKVError(status, msg)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, dim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d)


def kv_store(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Write k[t], v[t] to the cache slot slot_mapping[t]; slots equal to -1 are skipped."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if k.shape != v.shape or k_cache.shape != v_cache.shape:
        raise ValueError("k/v or k_cache/v_cache shapes differ")
    T = k.shape[0]
    if slot_mapping.shape[0] != T or tuple(k.shape[1:]) != tuple(k_cache.shape[2:]):
        raise ValueError("shape mismatch between k, slot_mapping and the cache")
    _check(lib.pkv_kv_store(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                            k_cache.data_ptr(), v_cache.data_ptr(), _cache_desc(k_cache),
                            _stream_ptr(stream)))


def decode_plan(num_seqs: int, num_q_heads: int, k_cache: torch.Tensor, max_context_len: int,
                split_tokens: int = 0, engine: Optional[int] = None) -> DecodePlan:
    """Host-side decode plan (chunking, workspace size and engine); see pkv_decode_plan_make.
    engine: None keeps the library's choice (the tensor-core engine for head_dim 128,
    block_size >= 128 and >= 4 query heads per kv head, else the CUDA-core engine), or
    DECODE_ENGINE_CUDA_CORE / DECODE_ENGINE_TENSOR_CORE to override it."""
    plan = DecodePlan()
    _check(lib.pkv_decode_plan_make(num_seqs, num_q_heads, _cache_desc(k_cache),
                                    int(max_context_len), int(split_tokens), ctypes.byref(plan)))
    if engine is not None:
        plan.engine = int(engine)
    return plan


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _key_and_stream(device, stream):
    dev = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return (dev.index, s.cuda_stream), s


def workspace_for(plan: DecodePlan, device: torch.device, stream=None) -> torch.Tensor:
    """The default decode workspace of (device, stream): grow-only, uint8, 256-byte aligned by the
    caching allocator.

    Calls on one stream run in order, so they share it; calls on different streams get different
    workspaces and never race. The buffer is allocated on `stream` itself, so when it is replaced
    by a larger one the caching allocator hands its memory out again only to work on that stream,
    i.e. after the kernels that used it.
    """
    key, s = _key_and_stream(device, stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < plan.workspace_bytes:
            with torch.cuda.stream(s):
                ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8,
                                 device=key[0])
            _ws_cache[key] = ws
        return ws


def _reused(plan: Optional[DecodePlan]) -> DecodePlan:
    """A copy of plan with PKV_DECODE_PLAN_REUSE set (the caller's plan object is unchanged)."""
    if plan is None:
        raise ValueError("reuse_plan needs the plan of the earlier decode call")
    p = DecodePlan.from_buffer_copy(plan)
    p.flags |= DECODE_PLAN_REUSE
    return p


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, out=None,
                 max_context_len: Optional[int] = None, split_tokens: int = 0,
                 plan: Optional[DecodePlan] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None, engine: Optional[int] = None, reuse_plan: bool = False):
    """Decode attention over the paged cache. Returns out [num_seqs, num_q_heads, head_dim] bf16.

    max_context_len bounds context_lens (host int); if omitted it is read from the device (a
    synchronisation). split_tokens: 0 automatic, > 0 fixed chunk length, < 0 never split.
    reuse_plan: run on the device plan the previous call with this plan and workspace left
    (same lengths, e.g. the layers of a decode step after the first): no plan kernel.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    B, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes do not match q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch size differs from q")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if plan is None:
        if max_context_len is None:
            max_context_len = int(context_lens.max().item()) if B else 0
        plan = decode_plan(B, Hq, k_cache, max_context_len, split_tokens, engine)
    if workspace is None:
        workspace = workspace_for(plan, q.device, stream)
    if reuse_plan:
        plan = _reused(plan)
    _check(lib.pkv_paged_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                _cache_desc(k_cache), block_tables.data_ptr(),
                                block_tables.shape[1], context_lens.data_ptr(), B, Hq,
                                float(scale), ctypes.byref(plan), out.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)))
    return out


def paged_decode_store(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                       context_lens, scale: float, out=None, max_context_len: Optional[int] = None,
                       split_tokens: int = 0, plan: Optional[DecodePlan] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None,
                       engine: Optional[int] = None, reuse_plan: bool = False):
    """One decode step with the store fused in: writes k_new[b], v_new[b] to slot_mapping[b] and
    attends over context_lens[b] tokens, the last of which is taken from k_new / v_new.
    reuse_plan as for paged_decode (the store still runs, in a grid of its own)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    B, Hq, D = q.shape
    if (k_new.shape != (B,) + tuple(k_cache.shape[2:]) or v_new.shape != k_new.shape
            or slot_mapping.shape[0] != B):
        raise ValueError("k_new / v_new must be [num_seqs, Hkv, D] and slot_mapping [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    if plan is None:
        if max_context_len is None:
            max_context_len = int(context_lens.max().item()) if B else 0
        plan = decode_plan(B, Hq, k_cache, max_context_len, split_tokens, engine)
    if workspace is None:
        workspace = workspace_for(plan, q.device, stream)
    if reuse_plan:
        plan = _reused(plan)
    _check(lib.pkv_paged_decode_store(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                      slot_mapping.data_ptr(), k_cache.data_ptr(),
                                      v_cache.data_ptr(), _cache_desc(k_cache),
                                      block_tables.data_ptr(), block_tables.shape[1],
                                      context_lens.data_ptr(), B, Hq, float(scale),
                                      ctypes.byref(plan), out.data_ptr(), workspace.data_ptr(),
                                      workspace.numel(), _stream_ptr(stream)))
    return out


PREFILL_WORKSPACE_BYTES = 256  # PKV_PREFILL_WORKSPACE_BYTES
_prefill_ws: dict = {}


def prefill_workspace_bytes(num_seqs: int) -> int:
    """Workspace bytes with which paged_prefill numbers its work densely (no empty query tiles
    to skip); see pkv_prefill_workspace_bytes."""
    return int(lib.pkv_prefill_workspace_bytes(int(num_seqs)))


def prefill_workspace(device: torch.device, stream=None, num_seqs: int = 0) -> torch.Tensor:
    """The default prefill workspace of (device, stream), grow-only and allocated on that
    stream: calls on one stream share it in order, calls on different streams never race. It is
    sized for num_seqs sequences (dense work numbering)."""
    key, s = _key_and_stream(device, stream)
    need = prefill_workspace_bytes(num_seqs)
    with _ws_lock:
        ws = _prefill_ws.get(key)
        if ws is None or ws.numel() < need:
            with torch.cuda.stream(s):
                ws = torch.empty(need, dtype=torch.uint8, device=key[0])
            _prefill_ws[key] = ws
        return ws


def paged_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, block_tables, scale: float,
                  k_cache=None, v_cache=None, out=None, max_seqlen_q: Optional[int] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None):
    """Varlen causal prefill. With block_tables, every key is read through the table (store the
    new tokens with kv_store first); without, keys come from k and v and there is no prefix."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    Tq, Hq, D = q.shape
    B = cu_seqlens_q.shape[0] - 1
    if block_tables is not None:
        _need(block_tables, "block_tables", torch.int32, 2)
        _need(k_cache, "k_cache", torch.bfloat16, 4)
        _need(v_cache, "v_cache", torch.bfloat16, 4)
        desc = _cache_desc(k_cache)
        mb = block_tables.shape[1]
        bt_ptr, kc_ptr, vc_ptr = block_tables.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    else:
        desc = CacheDesc(1, 16, k.shape[1], D)
        mb, bt_ptr, kc_ptr, vc_ptr = 0, None, None, None
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    if workspace is None:
        workspace = prefill_workspace(q.device, stream, B)
    _check(lib.pkv_paged_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Tq,
                                 int(max_seqlen_q), bt_ptr, mb, kc_ptr, vc_ptr, desc, Hq,
                                 float(scale), out.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)))
    return out


def get_device_error() -> int:
    """Read and clear the device error word (PKV_DEVERR_* bits); synchronises the device."""
    v = ctypes.c_int32(0)
    _check(lib.pkv_get_device_error(ctypes.byref(v)))
    return int(v.value)


def selftest_bounded_wait(stream=None):
    """Run the bounded-wait diagnostic (about one second); returns the device error word."""
    _check(lib.pkv_selftest_bounded_wait(_stream_ptr(stream)))
    return get_device_error()


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """Copy-on-write: block pairs[i, 1] := block pairs[i, 0] in both caches."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(pairs, "pairs", torch.int32, 2)
    if pairs.shape[1] != 2 or k_cache.shape != v_cache.shape:
        raise ValueError("pairs must be [n, 2] and the caches alike")
    _check(lib.pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), _cache_desc(k_cache),
                               pairs.data_ptr(), pairs.shape[0], _stream_ptr(stream)))


def gather_blocks(k_cache, v_cache, ids, out_k=None, out_v=None, stream=None):
    """Swap out: returns (out_k, out_v) [n, block_size, Hkv, D] holding blocks ids of each cache."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(ids, "ids", torch.int32, 1)
    shape = (ids.shape[0],) + tuple(k_cache.shape[1:])
    out_k = torch.empty(shape, dtype=torch.bfloat16, device=k_cache.device) if out_k is None \
        else out_k
    out_v = torch.empty(shape, dtype=torch.bfloat16, device=k_cache.device) if out_v is None \
        else out_v
    _need(out_k, "out_k", torch.bfloat16, 4)
    _need(out_v, "out_v", torch.bfloat16, 4)
    _check(lib.pkv_gather_blocks(k_cache.data_ptr(), v_cache.data_ptr(), _cache_desc(k_cache),
                                 ids.data_ptr(), ids.shape[0], out_k.data_ptr(),
                                 out_v.data_ptr(), _stream_ptr(stream)))
    return out_k, out_v


def scatter_blocks(in_k, in_v, ids, k_cache, v_cache, stream=None):
    """Swap in: k_cache[ids[i]] := in_k[i], v_cache[ids[i]] := in_v[i]."""
    for t, name in ((in_k, "in_k"), (in_v, "in_v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, name, torch.bfloat16, 4)
    _need(ids, "ids", torch.int32, 1)
    _check(lib.pkv_scatter_blocks(in_k.data_ptr(), in_v.data_ptr(), ids.data_ptr(),
                                  ids.shape[0], k_cache.data_ptr(), v_cache.data_ptr(),
                                  _cache_desc(k_cache), _stream_ptr(stream)))


def block_hashes(token_ids, cu_seqlens, block_size: int, max_blocks: int, out=None, stream=None):
    """Chained xxhash64 of each sequence's full blocks: int64 tensor [num_seqs, max_blocks]
    holding the uint64 hash bits (0 where a sequence has no full block)."""
    _need(token_ids, "token_ids", torch.int32, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    B = cu_seqlens.shape[0] - 1
    if out is None:
        out = torch.empty((B, max_blocks), dtype=torch.int64, device=token_ids.device)
    _need(out, "out", torch.int64, 2)
    _check(lib.pkv_block_hashes(token_ids.data_ptr(), cu_seqlens.data_ptr(), B, int(block_size),
                                int(max_blocks), out.data_ptr(), _stream_ptr(stream)))
    return out
