"""Python binding of libpagedkv: decode-time paged attention for GB300.

Argument marshalling only. Every step of the path runs in the CUDA library
``libpagedkv.so`` (built in-tree by :func:`build`); there is no CPU or
PyTorch fallback, and every entry point raises if the library is missing.
The functions carry the C ABI's names (``include/pagedkv.h``):

* :func:`pk_reshape_and_cache` -- scatter new tokens' K/V into their slots;
* :func:`pk_copy_blocks` -- copy-on-write block copies;
* :func:`pk_paged_attention_decode` -- attention through the block tables,
  with optional split-K partitions merged by log-sum-exp;
* :class:`BlockManager` -- the host block manager (free list, refcounts,
  fork, copy-on-write, block tables, slot mappings).

PyTorch provides device memory and streams: the device entry points take
CUDA tensors and enqueue on the current stream unless one is given.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

from ._build import LIB_PATH, build

__all__ = [
    "build", "lib", "PagedKVError", "CacheDesc", "cache_desc",
    "pk_reshape_and_cache", "pk_reshape_and_cache_append", "pk_copy_blocks", "pk_paged_attention_decode",
    "pk_paged_attention_workspace_size", "pk_paged_attention_resolve_partition",
    "pk_get_device_error", "pk_status_string", "BlockManager",
    "PK_F32", "PK_BF16", "IMPLS", "DEVERR_NAMES",
]

PK_OK, PK_ERR_INVALID_ARG, PK_ERR_UNSUPPORTED, PK_ERR_OUT_OF_BLOCKS = 0, 1, 2, 3
PK_ERR_UNKNOWN_SEQ, PK_ERR_SEQ_EXISTS, PK_ERR_CUDA, PK_ERR_WORKSPACE = 4, 5, 6, 7
PK_ERR_INVARIANT, PK_ERR_NOMEM = 8, 9
PK_F32, PK_BF16 = 0, 1
IMPLS = {"auto": 0, "simt": 1, "mma": 2}
PK_STATIC_WORKSPACE_BYTES = 64 << 20  # the static split-K scratch of pk_paged_attention_decode_static
DEVERR_NAMES = {0: "none", 1: "slot", 2: "block_id", 3: "pair", 4: "context", 5: "timeout", 6: "order"}

# Every symbol include/pagedkv.h declares.
EXPORTED = (
    "pk_reshape_and_cache", "pk_reshape_and_cache_append", "pk_copy_blocks", "pk_paged_attention_decode",
    "pk_paged_attention_decode_impl", "pk_paged_attention_decode_static", "pk_paged_attention_decode_items",
    "pk_attention_work_items", "pk_attention_plan", "pk_paged_attention_decode_append",
    "pk_paged_attention_decode_advance", "pk_selftest_wait_timeout", "pk_read_stream",
    "pk_paged_attention_resolve_partition",
    "pk_paged_attention_workspace_size", "pk_longest_first_order", "pk_get_device_error", "pk_status_string",
    "pk_bm_create", "pk_bm_destroy", "pk_bm_add_seq", "pk_bm_append_slots", "pk_bm_append_batch",
    "pk_bm_fork", "pk_bm_free_seq", "pk_bm_seq_len", "pk_bm_block_table", "pk_bm_export_tables",
    "pk_bm_num_free", "pk_bm_refcount", "pk_bm_check_invariants", "pk_bm_stats",
    "pk_decode_step_meta_bytes", "pk_decode_step", "pk_decode_step_prepare", "pk_decode_step_launch",
    "pk_decode_step_graph_count", "pk_decode_step_release",
    "pk_bm_prefix_groups", "pk_cascade_attention_decode", "pk_cascade_workspace_size",
    "pk_swap_blocks", "pk_bm_set_swap_space", "pk_bm_swap_out", "pk_bm_swap_in", "pk_bm_is_swapped",
    "pk_bm_host_free", "pk_bm_add_seq_cached", "pk_bm_commit", "pk_bm_cache_match", "pk_bm_cache_stats",
    "pk_bm_is_cached", "pk_bm_free_blocks", "pk_sim_num_steps", "pk_sim_run",
)
PK_POLICY = {"max_reservation": 0, "exact_contiguous": 1, "paged": 2}
PK_SIM_RULE = {"drop": 0, "stall": 1}
PK_SWAP_OUT, PK_SWAP_IN = 0, 1


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class StepBuffers(ctypes.Structure):
    _fields_ = [("q_host", ctypes.c_void_p), ("k_host", ctypes.c_void_p), ("v_host", ctypes.c_void_p),
                ("q_dev", ctypes.c_void_p), ("k_dev", ctypes.c_void_p), ("v_dev", ctypes.c_void_p),
                ("meta_host", ctypes.c_void_p), ("meta_dev", ctypes.c_void_p), ("meta_bytes", ctypes.c_size_t),
                ("out_dev", ctypes.c_void_p), ("out_host", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("tables_resident", ctypes.c_int32), ("plan_partition", ctypes.c_int32),
                ("plan_items", ctypes.c_int32), ("state", ctypes.c_void_p)]


class SimRequest(ctypes.Structure):
    _fields_ = [("arrival", ctypes.c_int32), ("prompt", ctypes.c_int32), ("max_new", ctypes.c_int32),
                ("gen", ctypes.c_int32), ("completion", ctypes.c_int32)]


class SimSummary(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "admitted", "rejected", "rejected_despite_free", "growth_failures", "growth_failures_despite_free",
        "dropped", "completed", "peak_live", "peak_reserved", "peak_waste", "capacity")] + \
        [("num_steps", ctypes.c_int32)]


class SimSample(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("active", ctypes.c_int32)] + \
        [(n, ctypes.c_int64) for n in ("live", "reserved", "waste", "free_slots", "largest_free")]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {pk_status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libpagedkv; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpagedkv is not built ({LIB_PATH} missing): call "
                           "paged_kv_cache_113_gb300.build() first")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(CacheDesc)
    sigs = {
        "pk_reshape_and_cache": (i32, [P, P, P, i32, P, P, D, P]),
        "pk_reshape_and_cache_append": (i32, [P, P, P, i32, P, P, D, P, i32, P, P]),
        "pk_copy_blocks": (i32, [P, P, P, i32, D, P]),
        "pk_paged_attention_decode": (i32, [P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, i32, P, sz, D, P]),
        "pk_paged_attention_decode_impl": (i32, [P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, P, sz, D,
                                                 P, i32, P]),
        "pk_longest_first_order": (i32, [P, i32, P]),
        "pk_paged_attention_decode_items": (i32, [P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, P, i32, P, sz,
                                                  D, i32, P]),
        "pk_attention_work_items": (i32, [P, i32, i32, P, i32, P]),
        "pk_attention_plan": (i32, [P, i32, i32, i32, D, P, P, i32, P]),
        "pk_paged_attention_decode_append": (i32, [P, P, P, P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, P,
                                                   i32, P, sz, D, P]),
        "pk_selftest_wait_timeout": (i32, [ctypes.c_uint32, P]),
        "pk_read_stream": (i32, [P, sz, P, P]),
        "pk_paged_attention_decode_advance": (i32, [P, P, P, P, P, P, P, P, P, P, f32, i32, i32, i32, i32, i32,
                                                     P, i32, P, sz, D, P]),
        "pk_paged_attention_decode_static": (i32, [P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, i32, D, P]),
        "pk_paged_attention_resolve_partition": (i32, [i32, i32, i32, i32, D]),
        "pk_paged_attention_workspace_size": (sz, [i32, i32, i32, i32, D]),
        "pk_get_device_error": (i32, [P, P]),
        "pk_status_string": (ctypes.c_char_p, [i32]),
        "pk_bm_create": (i32, [i32, i32, P, P]),
        "pk_bm_destroy": (None, [P]),
        "pk_bm_add_seq": (i32, [P, i64]),
        "pk_bm_append_slots": (i32, [P, i64, i32, P, P, P]),
        "pk_bm_append_batch": (i32, [P, P, i32, P, P, P]),
        "pk_bm_fork": (i32, [P, i64, i64]),
        "pk_bm_free_seq": (i32, [P, i64]),
        "pk_bm_seq_len": (i32, [P, i64, P]),
        "pk_bm_block_table": (i32, [P, i64, P, i32, P]),
        "pk_bm_export_tables": (i32, [P, P, i32, i32, P, P]),
        "pk_bm_num_free": (i32, [P]),
        "pk_bm_refcount": (i32, [P, i32]),
        "pk_bm_check_invariants": (i32, [P]),
        "pk_bm_stats": (i32, [P, P, P, P, P, P]),
        "pk_decode_step_meta_bytes": (sz, [i32, i32]),
        "pk_bm_prefix_groups": (i32, [P, P, i32, i32, i32, P, P, P, P, P]),
        "pk_cascade_attention_decode": (i32, [P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, P, P, P, P,
                                              i32, i32, i32, P, P, sz, D, P]),
        "pk_cascade_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, D]),
        "pk_swap_blocks": (i32, [P, P, P, P, i32, P, i32, i32, D, P]),
        "pk_bm_set_swap_space": (i32, [P, i32, P]),
        "pk_bm_swap_out": (i32, [P, i64, P, i32, P]),
        "pk_bm_swap_in": (i32, [P, i64, P, i32, P]),
        "pk_bm_is_swapped": (i32, [P, i64]),
        "pk_bm_host_free": (i32, [P]),
        "pk_bm_add_seq_cached": (i32, [P, i64, P, i32, P]),
        "pk_bm_commit": (i32, [P, i64, P, i32]),
        "pk_bm_cache_match": (i32, [P, P, i32, P]),
        "pk_bm_cache_stats": (i32, [P, P, P, P, P]),
        "pk_bm_is_cached": (i32, [P, i32]),
        "pk_bm_free_blocks": (i32, [P, P, i32, P]),
        "pk_sim_num_steps": (i32, [P, i32]),
        "pk_sim_run": (i32, [P, i32, i32, i32, i32, i32, ctypes.POINTER(SimSummary), P, i32]),
        "pk_decode_step": (i32, [P, P, i32, i32, f32, i32, i32, P, P, D, ctypes.POINTER(StepBuffers), P]),
        "pk_decode_step_prepare": (i32, [P, P, i32, i32, i32, i32, D, ctypes.POINTER(StepBuffers)]),
        "pk_decode_step_launch": (i32, [i32, i32, f32, i32, P, P, D, ctypes.POINTER(StepBuffers), P]),
        "pk_decode_step_graph_count": (i32, [ctypes.POINTER(StepBuffers)]),
        "pk_decode_step_release": (None, [ctypes.POINTER(StepBuffers)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def pk_status_string(status: int) -> str:
    return lib().pk_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != PK_OK:
        raise PagedKVError(status, what)


# ---------------------------------------------------------------------------
# Device entry points (torch tensors)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return PK_F32
    if t.dtype == torch.bfloat16:
        return PK_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: libpagedkv takes float32 or bfloat16")


def cache_desc(k_cache) -> CacheDesc:
    """The pool descriptor of a ``[num_blocks, B, Hk, d]`` cache tensor."""
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [num_blocks, block_size, num_kv_heads, head_dim]")
    N, B, Hk, d = k_cache.shape
    return CacheDesc(int(N), int(B), int(Hk), int(d), _dtype_code(k_cache))


def _dev(t, name, dtype=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libpagedkv has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def pk_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Writes token i's K/V ``[T, Hk, d]`` into slot ``slot_mapping[i]`` (int64)."""
    torch = _torch()
    desc = cache_desc(k_cache)
    T = int(k.shape[0])
    if tuple(k.shape) != (T, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise ValueError("k and v must be [num_tokens, num_kv_heads, head_dim]")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("k, v, k_cache and v_cache must share one dtype")
    if v_cache.shape != k_cache.shape or tuple(slot_mapping.shape) != (T,):
        raise ValueError("shape mismatch")
    _check(lib().pk_reshape_and_cache(_dev(k, "k"), _dev(v, "v"), _dev(slot_mapping, "slot_mapping", torch.int64),
                                      T, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                      ctypes.byref(desc), _stream(stream)), "pk_reshape_and_cache")


def pk_reshape_and_cache_append(k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, stream=None):
    """Scatter of one decode step plus the device-side table update: row i's
    next token goes to ``slot_mapping[i]``, ``block_tables[i][ctx/B]`` becomes
    ``slot/B`` and ``context_lens[i]`` grows by one (int32 CUDA tensors)."""
    torch = _torch()
    desc = cache_desc(k_cache)
    T = int(k.shape[0])
    if slot_mapping.dtype != torch.int64 or block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("slot_mapping int64, block_tables and context_lens int32")
    if block_tables.shape[0] != T or context_lens.shape[0] != T or not block_tables.is_contiguous():
        raise ValueError("block_tables [T, max_blocks] and context_lens [T]")
    _check(lib().pk_reshape_and_cache_append(_dev(k, "k"), _dev(v, "v"), _dev(slot_mapping, "slot_mapping"), T,
                                             _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                             _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
                                             _dev(context_lens, "context_lens"), _stream(stream)),
           "pk_reshape_and_cache_append")


def pk_copy_blocks(k_cache, v_cache, src_dst_pairs, stream=None):
    """Copies whole blocks ``src_dst_pairs[p] = (src, dst)`` (int64 ``[n, 2]``) in K and V."""
    torch = _torch()
    desc = cache_desc(k_cache)
    n = int(src_dst_pairs.shape[0]) if src_dst_pairs.numel() else 0
    if n and tuple(src_dst_pairs.shape) != (n, 2):
        raise ValueError("src_dst_pairs must be [num_pairs, 2]")
    if n == 0:
        return
    _check(lib().pk_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                _dev(src_dst_pairs, "src_dst_pairs", torch.int64), n, ctypes.byref(desc),
                                _stream(stream)), "pk_copy_blocks")


def pk_paged_attention_resolve_partition(num_seqs, num_q_heads, max_context_len, partition_size, desc) -> int:
    return int(lib().pk_paged_attention_resolve_partition(int(num_seqs), int(num_q_heads), int(max_context_len),
                                                          int(partition_size), ctypes.byref(desc)))


def pk_paged_attention_workspace_size(num_seqs, num_q_heads, max_context_len, partition_size, desc) -> int:
    return int(lib().pk_paged_attention_workspace_size(int(num_seqs), int(num_q_heads), int(max_context_len),
                                                       int(partition_size), ctypes.byref(desc)))


def pk_longest_first_order(context_lens) -> np.ndarray:
    """Host helper: sequence indices by descending context length (ties by index)."""
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty(max(len(lens), 1), np.int32)
    _check(lib().pk_longest_first_order(_np_ptr(lens), len(lens), _np_ptr(out)), "pk_longest_first_order")
    return out[: len(lens)]


def pk_attention_work_items(context_lens, partition: int) -> np.ndarray:
    """Host helper: the (sequence, partition) work items, longest first, int32 [n, 2]."""
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    n = ctypes.c_int32(0)
    lib().pk_attention_work_items(_np_ptr(lens), len(lens), int(partition), None, 0, ctypes.byref(n))
    out = np.empty((max(n.value, 1), 2), np.int32)
    _check(lib().pk_attention_work_items(_np_ptr(lens), len(lens), int(partition), _np_ptr(out), n.value,
                                         ctypes.byref(n)), "pk_attention_work_items")
    return out[: n.value]


def pk_attention_plan(context_lens, num_q_heads: int, desc: CacheDesc, partition_size: int = -1):
    """Host planner: ``(partition, items int32 [n, 2])`` for the host context
    lengths (see pk_attention_plan in the header)."""
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    part, n = ctypes.c_int32(0), ctypes.c_int32(0)
    lib().pk_attention_plan(_np_ptr(lens), len(lens), int(num_q_heads), int(partition_size), ctypes.byref(desc),
                            ctypes.byref(part), None, 0, ctypes.byref(n))
    out = np.empty((max(n.value, 1), 2), np.int32)
    _check(lib().pk_attention_plan(_np_ptr(lens), len(lens), int(num_q_heads), int(partition_size),
                                   ctypes.byref(desc), ctypes.byref(part), _np_ptr(out), n.value, ctypes.byref(n)),
           "pk_attention_plan")
    return int(part.value), out[: n.value]


def pk_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                              max_context_len: int, partition_size: int = -1, workspace=None,
                              impl: str = "auto", stream=None, seq_order=None, work_items=None):
    """Decode attention through the block tables; writes ``out`` ``[S, Hq, d]``.

    ``block_tables`` int32 ``[S, max_blocks]``, ``context_lens`` int32 ``[S]``
    (lengths after the step token). ``partition_size``: 0 = no split, -1 =
    automatic, >0 = split-K partition in tokens. ``workspace``: a CUDA tensor
    of at least :func:`pk_paged_attention_workspace_size` bytes when the
    partitioning splits. ``seq_order``: optional int32 CUDA tensor ``[S]``, the
    launch order of the sequences (see :func:`pk_longest_first_order`).
    ``work_items``: optional int32 CUDA tensor ``[n, 2]`` of (sequence,
    partition) items for the resolved partition size (see
    :func:`pk_attention_work_items`); replaces ``seq_order``.
    """
    torch = _torch()
    desc = cache_desc(k_cache)
    S, Hq, d = (int(x) for x in q.shape)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out and q must be [num_seqs, num_q_heads, head_dim] of the cache dtype")
    if d != desc.head_dim or block_tables.dim() != 2 or int(block_tables.shape[0]) != S:
        raise ValueError("shape mismatch")
    if tuple(context_lens.shape) != (S,):
        raise ValueError("context_lens must be [num_seqs]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    if impl not in IMPLS:
        raise ValueError(f"impl must be one of {sorted(IMPLS)}")
    if work_items is not None:
        if work_items.dim() != 2 or int(work_items.shape[1]) != 2:
            raise ValueError("work_items must be [n, 2]")
        _check(lib().pk_paged_attention_decode_items(
            _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
            float(scale), S, Hq, int(block_tables.shape[1]), int(max_context_len), int(partition_size),
            _dev(work_items, "work_items", torch.int32), int(work_items.shape[0]), ws_ptr, ws_bytes,
            ctypes.byref(desc), IMPLS[impl], _stream(stream)), "pk_paged_attention_decode_items")
        return
    _check(lib().pk_paged_attention_decode_impl(
        _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        float(scale), S, Hq, int(block_tables.shape[1]), int(max_context_len), int(partition_size),
        ws_ptr, ws_bytes, ctypes.byref(desc),
        None if seq_order is None else _dev(seq_order, "seq_order", torch.int32),
        IMPLS[impl], _stream(stream)), "pk_paged_attention_decode")


def pk_paged_attention_decode_append(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                                     context_lens, scale: float, max_context_len: int, partition_size: int,
                                     work_items, workspace=None, stream=None):
    """A step's scatter fused into its attention (see the header): token i of
    ``k_new``/``v_new`` ``[S, Hk, d]`` goes to ``slot_mapping[i]`` and is
    sequence i's last token; ``work_items`` int32 ``[n, 2]`` for the given
    (resolved) partition size."""
    torch = _torch()
    desc = cache_desc(k_cache)
    S, Hq, d = (int(x) for x in q.shape)
    if out.shape != q.shape or tuple(k_new.shape) != (S, desc.num_kv_heads, d) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib().pk_paged_attention_decode_append(
        _dev(out, "out"), _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        float(scale), S, Hq, int(block_tables.shape[1]), int(max_context_len), int(partition_size),
        _dev(work_items, "work_items", torch.int32), int(work_items.shape[0]), ws_ptr, ws_bytes,
        ctypes.byref(desc), _stream(stream)), "pk_paged_attention_decode_append")


def pk_paged_attention_decode_advance(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                                      context_lens, context_lens_out, scale: float, max_context_len: int,
                                      partition_size: int, work_items, workspace=None, stream=None):
    """One step on device-resident tables (see the header): ``context_lens``
    are the lengths before the step's token, ``context_lens_out`` receives
    them plus one, ``block_tables`` is updated in place; ``max_context_len``
    and ``work_items`` are for the advanced lengths."""
    torch = _torch()
    desc = cache_desc(k_cache)
    S, Hq, d = (int(x) for x in q.shape)
    if out.shape != q.shape or tuple(k_new.shape) != (S, desc.num_kv_heads, d) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib().pk_paged_attention_decode_advance(
        _dev(out, "out"), _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        _dev(context_lens_out, "context_lens_out", torch.int32), float(scale), S, Hq,
        int(block_tables.shape[1]), int(max_context_len), int(partition_size),
        _dev(work_items, "work_items", torch.int32), int(work_items.shape[0]), ws_ptr, ws_bytes,
        ctypes.byref(desc), _stream(stream)), "pk_paged_attention_decode_advance")


def pk_paged_attention_decode_static(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                     max_context_len: int, partition_size: int = -1, stream=None):
    """As :func:`pk_paged_attention_decode`, for callers that cannot allocate
    device memory: the split-K scratch is the library's static device array
    (``PK_STATIC_WORKSPACE_BYTES``), shared by every call on a device, so
    calls whose work overlaps on the GPU race on it."""
    torch = _torch()
    desc = cache_desc(k_cache)
    S, Hq, d = (int(x) for x in q.shape)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out and q must be [num_seqs, num_q_heads, head_dim] of the cache dtype")
    if d != desc.head_dim or block_tables.dim() != 2 or int(block_tables.shape[0]) != S:
        raise ValueError("shape mismatch")
    _check(lib().pk_paged_attention_decode_static(
        _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        float(scale), int(desc.block_size), S, Hq, int(block_tables.shape[1]), int(max_context_len),
        int(partition_size), ctypes.byref(desc), _stream(stream)), "pk_paged_attention_decode_static")


def pk_cascade_workspace_size(num_seqs, num_q_heads, max_context_len, num_groups, max_prefix_len,
                              partition_size, desc) -> int:
    return int(lib().pk_cascade_workspace_size(int(num_seqs), int(num_q_heads), int(max_context_len),
                                               int(num_groups), int(max_prefix_len), int(partition_size),
                                               ctypes.byref(desc)))


def pk_cascade_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                max_context_len: int, groups: dict, partition_size: int = -1, workspace=None,
                                seq_order=None, stream=None):
    """Cascade (shared-prefix) decode attention; same result as
    :func:`pk_paged_attention_decode`. ``groups`` holds CUDA int32 tensors
    ``offsets``, ``members``, ``prefix_len``, ``seq_prefix_len`` and the ints
    ``num_groups``, ``max_group_size``, ``max_prefix_len`` (see
    :meth:`BlockManager.prefix_groups`)."""
    torch = _torch()
    desc = cache_desc(k_cache)
    S, Hq, d = (int(x) for x in q.shape)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out and q must be [num_seqs, num_q_heads, head_dim] of the cache dtype")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    i32 = torch.int32
    _check(lib().pk_cascade_attention_decode(
        _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", i32), _dev(context_lens, "context_lens", i32), float(scale), S, Hq,
        int(block_tables.shape[1]), int(max_context_len), int(partition_size),
        _dev(groups["offsets"], "offsets", i32), _dev(groups["members"], "members", i32),
        _dev(groups["prefix_len"], "prefix_len", i32), _dev(groups["seq_prefix_len"], "seq_prefix_len", i32),
        int(groups["num_groups"]), int(groups["max_group_size"]), int(groups["max_prefix_len"]),
        None if seq_order is None else _dev(seq_order, "seq_order", i32), ws_ptr, ws_bytes, ctypes.byref(desc),
        _stream(stream)), "pk_cascade_attention_decode")


def pk_swap_blocks(k_cache, v_cache, k_host, v_host, pairs, direction: int, stream=None):
    """Whole-block copies between the device pool and a pinned host pool
    ``[H, B, Hk, d]``: ``pairs`` int64 ``[n, 2]`` (CUDA or pinned CPU tensor)
    from pk_bm_swap_out (``PK_SWAP_OUT``) or pk_bm_swap_in (``PK_SWAP_IN``)."""
    desc = cache_desc(k_cache)
    if k_host.is_cuda or not k_host.is_pinned() or not v_host.is_pinned():
        raise ValueError("k_host and v_host must be pinned host tensors")
    if tuple(k_host.shape[1:]) != tuple(k_cache.shape[1:]) or v_host.shape != k_host.shape:
        raise ValueError("host pools must be [H, B, Hk, d] like the device pool")
    n = int(pairs.shape[0]) if pairs.numel() else 0
    if n == 0:
        return
    if pairs.dtype != _torch().int64 or not pairs.is_contiguous():
        raise TypeError("pairs must be contiguous int64 [n, 2]")
    if not (pairs.is_cuda or pairs.is_pinned()):
        raise ValueError("pairs must be a CUDA tensor or pinned host memory")
    _check(lib().pk_swap_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                ctypes.c_void_p(k_host.data_ptr()), ctypes.c_void_p(v_host.data_ptr()),
                                int(k_host.shape[0]), ctypes.c_void_p(pairs.data_ptr()), n, int(direction),
                                ctypes.byref(desc), _stream(stream)), "pk_swap_blocks")


def pk_get_device_error(stream=None) -> Tuple[int, int]:
    """Synchronises the stream, reads and clears the device error word.

    Returns ``(kind, index)``: kind 0 means no error (see DEVERR_NAMES).
    """
    code = ctypes.c_int32(0)
    _check(lib().pk_get_device_error(ctypes.byref(code), _stream(stream)), "pk_get_device_error")
    return code.value >> 24, code.value & 0xFFFFFF


# ---------------------------------------------------------------------------
# Host block manager
# ---------------------------------------------------------------------------
def _np_ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


class BlockManager:
    """Host block manager (``pk_bm_*``): free list, refcounts, fork, CoW."""

    def __init__(self, num_blocks: int, block_size: int, alloc_order: Optional[np.ndarray] = None):
        self._L = lib()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = None if alloc_order is None else np.ascontiguousarray(alloc_order, dtype=np.int32)
        if order is not None and order.shape != (self.num_blocks,):
            raise ValueError("alloc_order must hold num_blocks entries")
        h = ctypes.c_void_p()
        _check(self._L.pk_bm_create(self.num_blocks, self.block_size, _np_ptr(order), ctypes.byref(h)),
               "pk_bm_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._L.pk_bm_destroy(h)
            self._h = None

    def add_seq(self, seq: int):
        _check(self._L.pk_bm_add_seq(self._h, int(seq)), "pk_bm_add_seq")

    def append(self, seq: int, n: int):
        """Appends n tokens; returns (slots int64[n], (src, dst) CoW pair or None)."""
        slots = np.empty(max(int(n), 1), np.int64)
        pair = np.zeros(2, np.int64)
        ncow = ctypes.c_int32(0)
        _check(self._L.pk_bm_append_slots(self._h, int(seq), int(n), _np_ptr(slots), _np_ptr(pair),
                                          ctypes.byref(ncow)), "pk_bm_append_slots")
        return slots[: int(n)], ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def append_batch(self, seqs: Sequence[int]):
        """One token for each sequence in order; returns (slots [n], pairs [k, 2])."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = len(ids)
        slots = np.empty(max(n, 1), np.int64)
        pairs = np.empty((max(n, 1), 2), np.int64)
        ncow = ctypes.c_int32(0)
        _check(self._L.pk_bm_append_batch(self._h, _np_ptr(ids), n, _np_ptr(slots), _np_ptr(pairs),
                                          ctypes.byref(ncow)), "pk_bm_append_batch")
        return slots[:n], pairs[: ncow.value].copy()

    def fork(self, parent: int, child: int):
        _check(self._L.pk_bm_fork(self._h, int(parent), int(child)), "pk_bm_fork")

    def free_seq(self, seq: int):
        _check(self._L.pk_bm_free_seq(self._h, int(seq)), "pk_bm_free_seq")

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64(0)
        _check(self._L.pk_bm_seq_len(self._h, int(seq), ctypes.byref(n)), "pk_bm_seq_len")
        return int(n.value)

    def table(self, seq: int) -> np.ndarray:
        n = ctypes.c_int32(0)
        _check(self._L.pk_bm_block_table(self._h, int(seq), None, 0, ctypes.byref(n)), "pk_bm_block_table")
        out = np.empty(max(n.value, 1), np.int32)
        _check(self._L.pk_bm_block_table(self._h, int(seq), _np_ptr(out), n.value, ctypes.byref(n)),
               "pk_bm_block_table")
        return out[: n.value]

    def export_tables(self, seqs: Sequence[int], max_blocks: int,
                      tables_out: Optional[np.ndarray] = None, lens_out: Optional[np.ndarray] = None):
        """Padded int32 tables ``[n, max_blocks]`` (pad -1) and int32 lengths ``[n]``."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = len(ids)
        tables = np.empty((n, max_blocks), np.int32) if tables_out is None else tables_out
        lens = np.empty(n, np.int32) if lens_out is None else lens_out
        assert tables.dtype == np.int32 and tables.flags.c_contiguous and tables.shape == (n, max_blocks)
        assert lens.dtype == np.int32 and lens.shape == (n,)
        _check(self._L.pk_bm_export_tables(self._h, _np_ptr(ids), n, int(max_blocks), _np_ptr(tables),
                                           _np_ptr(lens)), "pk_bm_export_tables")
        return tables, lens

    def set_swap_space(self, num_host_blocks: int, host_order: Optional[np.ndarray] = None):
        order = None if host_order is None else np.ascontiguousarray(host_order, dtype=np.int32)
        _check(self._L.pk_bm_set_swap_space(self._h, int(num_host_blocks), _np_ptr(order)), "pk_bm_set_swap_space")

    def _swap(self, fn, name, seq):
        n = len(self.table(seq))
        pairs = np.zeros((max(n, 1), 2), np.int64)
        cnt = ctypes.c_int32(0)
        _check(fn(self._h, int(seq), _np_ptr(pairs), n, ctypes.byref(cnt)), name)
        return pairs[: cnt.value]

    def swap_out(self, seq: int) -> np.ndarray:
        """(device block, host block) pairs, int64 [n, 2], in table order."""
        return self._swap(self._L.pk_bm_swap_out, "pk_bm_swap_out", seq)

    def swap_in(self, seq: int) -> np.ndarray:
        """(host block, device block) pairs, int64 [n, 2], in table order."""
        return self._swap(self._L.pk_bm_swap_in, "pk_bm_swap_in", seq)

    def is_swapped(self, seq: int) -> bool:
        return int(self._L.pk_bm_is_swapped(self._h, int(seq))) == 1

    def host_free(self) -> int:
        return int(self._L.pk_bm_host_free(self._h))

    # -- prefix caching -------------------------------------------------------
    def add_seq_cached(self, seq: int, tokens) -> int:
        """New sequence whose prompt is ``tokens`` (int32 ids); starts with the
        leading full blocks found in the cache. Returns the cached token count."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(self._L.pk_bm_add_seq_cached(self._h, int(seq), _np_ptr(t) if len(t) else None, len(t),
                                            ctypes.byref(n)), "pk_bm_add_seq_cached")
        return int(n.value)

    def commit(self, seq: int, tokens):
        """Registers the sequence's full blocks among ``tokens`` (its token ids)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(self._L.pk_bm_commit(self._h, int(seq), _np_ptr(t) if len(t) else None, len(t)), "pk_bm_commit")

    def cache_match(self, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(self._L.pk_bm_cache_match(self._h, _np_ptr(t) if len(t) else None, len(t), ctypes.byref(n)),
               "pk_bm_cache_match")
        return int(n.value)

    def cache_stats(self) -> dict:
        v = [ctypes.c_int64(0) for _ in range(4)]
        _check(self._L.pk_bm_cache_stats(self._h, *[ctypes.byref(x) for x in v]), "pk_bm_cache_stats")
        return dict(zip(("cached", "unreferenced", "hits", "evictions"), (int(x.value) for x in v)))

    def is_cached(self, block: int) -> bool:
        return int(self._L.pk_bm_is_cached(self._h, int(block))) == 1

    def free_blocks(self) -> np.ndarray:
        """The free list, next block to be handed out first."""
        n = ctypes.c_int32(0)
        _check(self._L.pk_bm_free_blocks(self._h, None, 0, ctypes.byref(n)), "pk_bm_free_blocks")
        out = np.empty(max(n.value, 1), np.int32)
        _check(self._L.pk_bm_free_blocks(self._h, _np_ptr(out), n.value, ctypes.byref(n)), "pk_bm_free_blocks")
        return out[: n.value]

    def prefix_groups(self, seqs: Sequence[int], max_group_size: int, min_prefix_blocks: int = 1) -> dict:
        """Shared-prefix groups of the batch ``seqs`` (host numpy arrays)."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = len(ids)
        offsets = np.zeros(n + 1, np.int32)
        members = np.zeros(max(n, 1), np.int32)
        prefix = np.zeros(max(n, 1), np.int32)
        seq_prefix = np.zeros(max(n, 1), np.int32)
        ng = ctypes.c_int32(0)
        _check(self._L.pk_bm_prefix_groups(self._h, _np_ptr(ids), n, int(max_group_size), int(min_prefix_blocks),
                                           _np_ptr(offsets), _np_ptr(members), _np_ptr(prefix), _np_ptr(seq_prefix),
                                           ctypes.byref(ng)), "pk_bm_prefix_groups")
        g = ng.value
        return {"num_groups": g, "offsets": offsets[: g + 1].copy(), "members": members[: offsets[g]].copy(),
                "prefix_len": prefix[:g].copy(), "seq_prefix_len": seq_prefix[:n].copy(),
                "max_group_size": int(max_group_size),
                "max_prefix_len": int(prefix[:g].max()) if g else 0}

    def num_free(self) -> int:
        return int(self._L.pk_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._L.pk_bm_refcount(self._h, int(block)))

    def check_invariants(self):
        _check(self._L.pk_bm_check_invariants(self._h), "pk_bm_check_invariants")

    def stats(self) -> dict:
        live, res, waste, cow = (ctypes.c_int64(0) for _ in range(4))
        shared = ctypes.c_int32(0)
        _check(self._L.pk_bm_stats(self._h, ctypes.byref(live), ctypes.byref(res), ctypes.byref(waste),
                                   ctypes.byref(shared), ctypes.byref(cow)), "pk_bm_stats")
        return {"live_tokens": live.value, "reserved_slots": res.value, "tail_waste": waste.value,
                "shared_blocks": shared.value, "cow_copies": cow.value}


class DecodeStepper:
    """Runs whole decode steps from pinned host buffers through pk_decode_step.

    Owns the pinned host staging (queries, new K/V, metadata, output) and the
    device buffers of one batch shape. ``step()`` calls pk_decode_step (host
    append, one metadata transfer, the kernels, the output copy) and
    synchronises; the output is then in ``out_host``. After the first step the
    block tables stay resident on the device and each step uploads only its
    slots and copy-on-write pairs; ``invalidate()`` forces a full upload.
    Steps run on the stepper's own stream (``stream``), where steady steps
    replay a captured CUDA graph; the first step, and the first after
    ``invalidate()``, wait for the caller's current stream. ``zero_copy``: the
    kernels read the inputs from, and write the output to, the stepper's
    pinned host buffers directly (fill ``q_host``/``k_host``/``v_host`` before
    each step).

    ``prepare()`` and ``launch_prepared()`` are the two halves of a step
    (pk_decode_step_prepare / pk_decode_step_launch): preparing step t+1
    right after launching step t overlaps its host work with step t on the
    GPU. Leave the block manager alone between a prepare and its launch;
    other changes to it (fork, free, swap) go between steps, followed by
    ``invalidate()``.
    """

    def __init__(self, bm: "BlockManager", seq_ids, num_q_heads: int, scale: float, max_blocks_per_seq: int,
                 k_cache, v_cache, partition_size: int = -1, max_context_len: Optional[int] = None,
                 zero_copy: bool = False):
        torch = _torch()
        self.bm, self.k_cache, self.v_cache = bm, k_cache, v_cache
        self.desc = cache_desc(k_cache)
        self.ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        S, Hk, d = len(self.ids), self.desc.num_kv_heads, self.desc.head_dim
        self.S, self.Hq, self.scale, self.maxb, self.partition = S, int(num_q_heads), float(scale), \
            int(max_blocks_per_seq), int(partition_size)
        dt, dev = k_cache.dtype, k_cache.device
        self.stream = torch.cuda.Stream(device=dev)
        self._order_after_caller = True
        self.q_host = torch.empty((S, self.Hq, d), dtype=dt).pin_memory()
        self.k_host = torch.empty((S, Hk, d), dtype=dt).pin_memory()
        self.v_host = torch.empty((S, Hk, d), dtype=dt).pin_memory()
        self.out_host = torch.empty((S, self.Hq, d), dtype=dt).pin_memory()
        # Zero-copy: the kernels read the inputs from, and write the output to,
        # the pinned host buffers directly (no device copies).
        self.zero_copy = bool(zero_copy)
        if self.zero_copy:
            self.q_dev = self.k_dev = self.v_dev = self.out_dev = None
        else:
            self.q_dev = torch.empty_like(self.q_host, device=dev)
            self.k_dev = torch.empty_like(self.k_host, device=dev)
            self.v_dev = torch.empty_like(self.v_host, device=dev)
            self.out_dev = torch.empty_like(self.out_host, device=dev)
        mb = int(lib().pk_decode_step_meta_bytes(S, self.maxb))
        self.meta_host = torch.empty(mb, dtype=torch.uint8).pin_memory()
        self.meta_dev = torch.empty(mb, dtype=torch.uint8, device=dev)
        mc = self.maxb * self.desc.block_size if max_context_len is None else int(max_context_len)
        # The automatic plan may choose any partition of at least 512 tokens.
        wsb = pk_paged_attention_workspace_size(S, self.Hq, mc, 512 if self.partition == -1 else self.partition,
                                                self.desc)
        self.workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
        ptr = lambda t: None if t is None else t.data_ptr()
        self.buffers = StepBuffers(
            self.q_host.data_ptr(), self.k_host.data_ptr(), self.v_host.data_ptr(),
            ptr(self.q_dev), ptr(self.k_dev), ptr(self.v_dev),
            self.meta_host.data_ptr(), self.meta_dev.data_ptr(), mb,
            ptr(self.out_dev), self.out_host.data_ptr(),
            None if self.workspace is None else self.workspace.data_ptr(), wsb)
        qkv = (self.q_host.numel() + self.k_host.numel() + self.v_host.numel()) * self.q_host.element_size()
        # Host -> device bytes of a step: the whole metadata buffer on a full
        # upload; only the slot section (plus 16 bytes per copy-on-write pair)
        # once the tables are resident.
        self.h2d_bytes_full = qkv + mb // 2     # one staging half
        self.h2d_bytes_resident = qkv + (8 * S + 255) // 256 * 256   # + the work list when it changes
        self.h2d_bytes = self.h2d_bytes_full
        # The call's arguments that never change, built once.
        self._step_fn = lib().pk_decode_step
        self._step_args = (bm._h, _np_ptr(self.ids), S, self.Hq, self.scale, self.maxb, self.partition,
                           ctypes.c_void_p(k_cache.data_ptr()), ctypes.c_void_p(v_cache.data_ptr()),
                           ctypes.byref(self.desc), ctypes.byref(self.buffers))
        self._stream_arg = ctypes.c_void_p(self.stream.cuda_stream)
        self._own_inputs = True  # the buffers struct points at q_host / k_host / v_host
        self._prepare_fn = lib().pk_decode_step_prepare
        self._prepare_args = (bm._h, _np_ptr(self.ids), S, self.Hq, self.maxb, self.partition,
                              ctypes.byref(self.desc), ctypes.byref(self.buffers))
        self._launch_fn = lib().pk_decode_step_launch
        self._launch_args = (S, self.Hq, self.scale, self.maxb, ctypes.c_void_p(k_cache.data_ptr()),
                             ctypes.c_void_p(v_cache.data_ptr()), ctypes.byref(self.desc),
                             ctypes.byref(self.buffers))
        self.d2h_bytes = self.out_host.numel() * self.out_host.element_size()

    def _bind(self, stream, q_host, k_host, v_host):
        if q_host is None and k_host is None and v_host is None:
            if not self._own_inputs:  # back to the stepper's own buffers
                for name in ("q_host", "k_host", "v_host"):
                    setattr(self.buffers, name, getattr(self, name).data_ptr())
                self._own_inputs = True
        else:
            for name, t in (("q_host", q_host), ("k_host", k_host), ("v_host", v_host)):
                setattr(self.buffers, name, (getattr(self, name) if t is None else t).data_ptr())
            self._own_inputs = False
        if self._order_after_caller:
            # Work the caller enqueued before (the prefill, a copy after a
            # fork) must finish before the step's kernels touch the pool.
            self.stream.wait_stream(_torch().cuda.current_stream())
            self._order_after_caller = False
        return self._stream_arg if stream is None else _stream(stream)

    def launch(self, stream=None, q_host=None, k_host=None, v_host=None):
        """Enqueues one step from q_host/k_host/v_host (the stepper's own pinned
        buffers unless other pinned tensors are given) on ``stream`` (default:
        the stepper's own stream, on which steady steps replay a captured graph)."""
        st = self._bind(stream, q_host, k_host, v_host)
        _check(self._step_fn(*self._step_args, st), "pk_decode_step")

    def prepare(self):
        """The host half of the next step (block-manager append, metadata);
        may run while the previous step is still on the GPU."""
        _check(self._prepare_fn(*self._prepare_args), "pk_decode_step_prepare")

    def launch_prepared(self, stream=None, q_host=None, k_host=None, v_host=None):
        """Enqueues the prepared step (arguments as ``launch``)."""
        st = self._bind(stream, q_host, k_host, v_host)
        _check(self._launch_fn(*self._launch_args, st), "pk_decode_step_launch")

    @property
    def graph_count(self) -> int:
        """Captured graphs the stepper holds (one per staging half at most)."""
        return int(lib().pk_decode_step_graph_count(ctypes.byref(self.buffers)))

    def release(self):
        """Frees the captured graphs (the stepper stays usable)."""
        if getattr(self, "buffers", None) is not None and self.buffers.state:
            lib().pk_decode_step_release(ctypes.byref(self.buffers))

    def __del__(self):
        try:
            self.release()
        except Exception:
            pass

    def invalidate(self):
        """The next step exports and uploads the whole tables again (call it
        after any block-manager change outside the stepper: fork, free, swap).
        The next step is also ordered after the caller's current stream."""
        self.buffers.tables_resident = 0
        self._order_after_caller = True

    def step(self, stream=None):
        """One step and a stream synchronise; returns the host output tensor."""
        self.launch(stream)
        (self.stream if stream is None else stream).synchronize()
        return self.out_host


# ---------------------------------------------------------------------------
# Allocator policy simulator
# ---------------------------------------------------------------------------
def pk_sim_run(trace, capacity: int, policy: str, block_size: int = 0, rule: str = "drop") -> dict:
    """Replays ``trace`` (dicts with arrival, prompt, max_new, gen, completion)
    under ``policy`` ("max_reservation", "exact_contiguous", "paged").
    Returns ``{"summary": dict, "samples": list of dicts}`` (one sample per step)."""
    L = lib()
    arr = (SimRequest * max(len(trace), 1))()
    for k, r in enumerate(trace):
        arr[k] = SimRequest(int(r["arrival"]), int(r["prompt"]), int(r["max_new"]), int(r["gen"]),
                            int(r["completion"]))
    steps = int(L.pk_sim_num_steps(arr, len(trace)))
    if steps < 0:
        raise ValueError("malformed trace")
    samples = (SimSample * max(steps, 1))()
    summ = SimSummary()
    _check(L.pk_sim_run(arr, len(trace), int(capacity), PK_POLICY[policy], int(block_size), PK_SIM_RULE[rule],
                        ctypes.byref(summ), samples, steps), "pk_sim_run")
    summary = {name: int(getattr(summ, name)) for name, _ in SimSummary._fields_}
    out = [{name: int(getattr(samples[t], name)) for name, _ in SimSample._fields_} for t in range(steps)]
    return {"summary": summary, "samples": out}
