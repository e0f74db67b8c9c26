"""CPU oracle for paged-KV-cache decode: TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The product path never does. The
oracle shares no code with the CUDA library: its arithmetic lives in
``oracle.c`` (plain single-threaded C, double precision), compiled here with
gcc into ``liboracle.so`` and called through ctypes.

What each function restates is documented in ``oracle.c``. The replay helper
:func:`run_workload` drives the oracle block manager through a workload's
host-operation plan, writes the pool with the oracle scatter / copy, then
runs one decode step (append one token per sequence, copy-on-write copies,
scatter, attention).

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` and ``tests/test_oracle_block_manager.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_OUT_OF_BLOCKS, ERR_UNKNOWN_SEQ, ERR_SEQ_EXISTS, ERR_NOMEM = range(6)
F32, BF16 = 0, 1


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, -O2, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                           check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # A test may point the loader at a deliberately broken build of oracle.c
    # (tests/test_oracle_mutants.py) to show that the pins catch it.
    override = os.environ.get("PKV_ORACLE_LIB")
    if override:
        lib = ctypes.CDLL(override)
    else:
        build()
        lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
    sig = {
        "or_bm_new": (P, [i32, i32, P]),
        "or_bm_delete": (None, [P]),
        "or_bm_add_seq": (i32, [P, i64]),
        "or_bm_append": (i32, [P, i64, i32, P, P, P]),
        "or_bm_fork": (i32, [P, i64, i64]),
        "or_bm_free_seq": (i32, [P, i64]),
        "or_bm_table": (i32, [P, i64, P, i32]),
        "or_bm_seq_len": (i64, [P, i64]),
        "or_bm_refcount": (i32, [P, i32]),
        "or_bm_num_free": (i32, [P]),
        "or_bm_cow_copies": (i64, [P]),
        "or_bm_free_list": (i32, [P, P, i32]),
        "or_bm_set_swap_space": (i32, [P, i32, P]),
        "or_bm_swap_out": (i32, [P, i64, P, P]),
        "or_bm_swap_in": (i32, [P, i64, P, P]),
        "or_bm_is_swapped": (i32, [P, i64]),
        "or_bm_host_free": (i32, [P]),
        "or_bm_add_seq_cached": (i32, [P, i64, P, i32, P]),
        "or_bm_commit": (i32, [P, i64, P, i32]),
        "or_bm_cache_stats": (None, [P, P, P, P, P]),
        "or_bm_is_cached": (i32, [P, i32]),
        "or_swap_copy": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32]),
        "or_reshape_and_cache": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32]),
        "or_copy_blocks": (i32, [P, P, P, i32, i32, i32, i32, i32, i32]),
        "or_paged_attention": (i32, [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32, i32, f64, P, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


class BlockManager:
    """The oracle's block manager (free list, refcounts, fork, CoW, free)."""

    def __init__(self, num_blocks: int, block_size: int, alloc_order: Optional[np.ndarray] = None):
        self._lib = _load()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = None
        if alloc_order is not None:
            order = np.ascontiguousarray(alloc_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("alloc_order must be a permutation of the pool")
        self._keep = order
        self._h = self._lib.or_bm_new(self.num_blocks, self.block_size, _ptr(order))
        if not self._h:
            raise OracleError(ERR_ARG, "or_bm_new")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.or_bm_delete(h)
            self._h = None

    def add_seq(self, seq: int):
        _check(self._lib.or_bm_add_seq(self._h, int(seq)), "add_seq")

    def append(self, seq: int, n: int):
        """Append n tokens; returns (slots int64[n], cow pair tuple or None)."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        cow = np.zeros(2, dtype=np.int64)
        ncow = ctypes.c_int(0)
        _check(self._lib.or_bm_append(self._h, int(seq), int(n), _ptr(slots), _ptr(cow),
                                      ctypes.byref(ncow)), "append")
        return slots[:n], ((int(cow[0]), int(cow[1])) if ncow.value else None)

    def fork(self, parent: int, child: int):
        _check(self._lib.or_bm_fork(self._h, int(parent), int(child)), "fork")

    def free_seq(self, seq: int):
        _check(self._lib.or_bm_free_seq(self._h, int(seq)), "free_seq")

    def table(self, seq: int) -> np.ndarray:
        n = self._lib.or_bm_table(self._h, int(seq), None, 0)
        if n < 0:
            raise OracleError(-n, "table")
        out = np.empty(max(n, 1), dtype=np.int32)
        self._lib.or_bm_table(self._h, int(seq), _ptr(out), n)
        return out[:n]

    def seq_len(self, seq: int) -> int:
        n = self._lib.or_bm_seq_len(self._h, int(seq))
        if n < 0:
            raise OracleError(ERR_UNKNOWN_SEQ, "seq_len")
        return int(n)

    def refcount(self, block: int) -> int:
        return int(self._lib.or_bm_refcount(self._h, int(block)))

    def num_free(self) -> int:
        return int(self._lib.or_bm_num_free(self._h))

    def cow_copies(self) -> int:
        return int(self._lib.or_bm_cow_copies(self._h))

    def free_list(self) -> np.ndarray:
        """The free stack, next block to be handed out first (cached blocks
        that no table names are not on it)."""
        n = int(self._lib.or_bm_free_list(self._h, None, 0))
        out = np.empty(max(n, 1), dtype=np.int32)
        self._lib.or_bm_free_list(self._h, _ptr(out), n)
        return out[:n]

    def set_swap_space(self, num_host_blocks: int, host_order: Optional[np.ndarray] = None):
        order = None if host_order is None else np.ascontiguousarray(host_order, dtype=np.int32)
        self._keep_host = order
        _check(self._lib.or_bm_set_swap_space(self._h, int(num_host_blocks), _ptr(order)), "set_swap_space")

    def swap_out(self, seq: int) -> np.ndarray:
        """(device block, host block) pairs, int64 [n, 2], in table order."""
        n = len(self.table(seq))
        pairs = np.zeros((max(n, 1), 2), np.int64)
        cnt = ctypes.c_int(0)
        _check(self._lib.or_bm_swap_out(self._h, int(seq), _ptr(pairs), ctypes.byref(cnt)), "swap_out")
        return pairs[: cnt.value]

    def swap_in(self, seq: int) -> np.ndarray:
        """(host block, device block) pairs, int64 [n, 2], in table order."""
        n = len(self.table(seq))
        pairs = np.zeros((max(n, 1), 2), np.int64)
        cnt = ctypes.c_int(0)
        _check(self._lib.or_bm_swap_in(self._h, int(seq), _ptr(pairs), ctypes.byref(cnt)), "swap_in")
        return pairs[: cnt.value]

    def is_swapped(self, seq: int) -> bool:
        return self._lib.or_bm_is_swapped(self._h, int(seq)) == 1

    def host_free(self) -> int:
        return int(self._lib.or_bm_host_free(self._h))

    # -- prefix caching ("PagedAttention" S06, "What's next") ----------------
    def add_seq_cached(self, seq: int, tokens) -> int:
        """New sequence whose prompt is ``tokens``; starts with every leading
        full block found in the cache. Returns the number of cached tokens."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int(0)
        _check(self._lib.or_bm_add_seq_cached(self._h, int(seq), _ptr(t) if len(t) else None, len(t),
                                              ctypes.byref(n)), "add_seq_cached")
        return int(n.value)

    def commit(self, seq: int, tokens):
        """Registers the sequence's full blocks among ``tokens`` (its token ids)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(self._lib.or_bm_commit(self._h, int(seq), _ptr(t) if len(t) else None, len(t)), "commit")

    def cache_stats(self) -> dict:
        v = [ctypes.c_longlong(0) for _ in range(4)]
        self._lib.or_bm_cache_stats(self._h, *[ctypes.byref(x) for x in v])
        return dict(zip(("cached", "unreferenced", "hits", "evictions"), (int(x.value) for x in v)))

    def is_cached(self, block: int) -> bool:
        return self._lib.or_bm_is_cached(self._h, int(block)) == 1

    def export_tables(self, seqs: Sequence[int], max_blocks: int) -> np.ndarray:
        """Padded ``int32 [len(seqs), max_blocks]`` tables, pad value -1."""
        out = np.full((len(seqs), max_blocks), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = self.table(s)
            if len(t) > max_blocks:
                raise ValueError("table longer than max_blocks")
            out[i, : len(t)] = t
        return out


def reshape_and_cache(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
                      slots: np.ndarray, num_blocks: int, block_size: int):
    """Write each token's K/V into its slot of the pool ``[N, B, Hk, d]`` (in place)."""
    lib = _load()
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    _, _, Hk, d = k_cache.shape
    _check(lib.or_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), _ptr(slots),
                                    int(len(slots)), int(num_blocks), int(block_size), int(Hk), int(d),
                                    int(k_cache.itemsize)), "reshape_and_cache")


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs: np.ndarray):
    """Copy whole blocks ``pairs[i] = (src, dst)`` of K and V (in place)."""
    lib = _load()
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    N, B, Hk, d = k_cache.shape
    _check(lib.or_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), int(len(pairs)), int(N), int(B),
                              int(Hk), int(d), int(k_cache.itemsize)), "copy_blocks")


def swap_copy(to_k: np.ndarray, to_v: np.ndarray, from_k: np.ndarray, from_v: np.ndarray, pairs: np.ndarray):
    """Whole-block copies between two pools: block pairs[i, 0] of `from` to pairs[i, 1] of `to`."""
    lib = _load()
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    _, B, Hk, d = to_k.shape
    _check(lib.or_swap_copy(_ptr(to_k), _ptr(to_v), _ptr(from_k), _ptr(from_v), _ptr(pairs), int(len(pairs)),
                            int(to_k.shape[0]), int(from_k.shape[0]), int(B), int(Hk), int(d), int(to_k.itemsize)),
           "swap_copy")


def paged_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, tables: np.ndarray,
                    ctx_lens: np.ndarray, scale: float, dtype: str,
                    select: Optional[np.ndarray] = None) -> np.ndarray:
    """Double-precision decode attention through the block tables.

    ``q`` is ``[S, Hq, d]`` (float32, or bf16 bits as uint16), the pools are
    ``[N, B, Hk, d]`` of the same storage type, ``tables`` ``int32 [S, maxb]``
    and ``ctx_lens`` ``[S]``. Returns ``float64 [S, Hq, d]``; with ``select``
    (``int32 [n, 2]`` rows of (seq, head)) only those rows are filled and the
    rest stay NaN.
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int64)
    S, Hq, d = q.shape
    N, B, Hk, d2 = k_cache.shape
    assert d2 == d
    out = np.full((S, Hq, d), np.nan, dtype=np.float64)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.int32).reshape(-1, 2)
    code = F32 if dtype == "f32" else BF16
    _check(lib.or_paged_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), code, _ptr(tables),
                                  int(tables.shape[1]), _ptr(ctx), int(S), int(Hq), int(Hk), int(d), int(B),
                                  int(N), float(scale), _ptr(sel), 0 if sel is None else int(len(sel))),
           "paged_attention")
    return out


def run_workload(wl, step: int = 0, attention: bool = True, select: Optional[np.ndarray] = None,
                 pool: bool = True) -> Dict[str, object]:
    """Replay a workload through the oracle and run one decode step.

    Returns a dict with the block manager ``bm``, the prefill slot mappings
    and CoW pairs in op order, the step's ``slots`` and ``cow_pairs``, the
    padded ``tables`` and ``ctx_lens`` after the step, the pools (if
    ``pool``) and the attention output ``out`` (float64, if ``attention``).
    :func:`continue_workload` runs further steps on the result.
    """
    from workloads import prefill_plan  # seeded inputs only

    bm = BlockManager(wl.num_blocks, wl.block_size, wl.alloc_order())
    shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc = np.zeros(shape, dtype=wl.np_dtype) if pool else None
    vc = np.zeros(shape, dtype=wl.np_dtype) if pool else None
    prefill_slots, prefill_pairs = [], []
    for op in prefill_plan(wl):
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        elif op[0] == "free":
            bm.free_seq(op[1])
        elif op[0] == "admit":
            # A request arrives: its prompt's leading full blocks come from the
            # prefix cache, the rest is written, then its full blocks are registered.
            r = op[1]
            toks = wl.chat_tokens(r)
            n_cached = bm.add_seq_cached(r, toks)
            if len(toks) > n_cached:
                slots, _ = bm.append(r, len(toks) - n_cached)
                prefill_slots.append(slots)
                if pool:
                    k, v = wl.chat_kv(r, n_cached, len(toks))
                    reshape_and_cache(kc, vc, k, v, slots, wl.num_blocks, wl.block_size)
            bm.commit(r, toks)
        else:
            _, seq, n, src = op
            slots, cow = bm.append(seq, n)
            prefill_slots.append(slots)
            if cow is not None:
                prefill_pairs.append(cow)
            if pool:
                if cow is not None:
                    copy_blocks(kc, vc, np.array([cow]))
                if src[0] == "prefix":
                    k, v = wl.prefix_kv(src[1])
                else:
                    k, v = wl.prefill_kv(src[1], n)
                reshape_and_cache(kc, vc, k, v, slots, wl.num_blocks, wl.block_size)
    res = {"bm": bm, "prefill_slots": prefill_slots, "prefill_pairs": prefill_pairs, "k_cache": kc, "v_cache": vc}
    return continue_workload(res, wl, step, attention=attention, select=select)


def continue_workload(res: Dict[str, object], wl, step: int, attention: bool = True,
                      select: Optional[np.ndarray] = None) -> Dict[str, object]:
    """One more decode step on the state a replay left in ``res``.

    In place: every sequence's length grows by one in index order (the
    append routine), the step's copy-on-write pairs are copied, the step's
    K/V (``wl.step_inputs(step)``) are scattered into their slots, and --
    with ``attention`` -- the step's attention is computed. ``res`` gets the
    step's ``slots``, ``cow_pairs``, padded ``tables``, ``ctx_lens``, inputs and
    ``out``; calling it again with the next step index continues the decode.
    """
    bm, kc, vc = res["bm"], res["k_cache"], res["v_cache"]
    pool = kc is not None
    q, kn, vn = wl.step_inputs(step)
    step_slots = np.empty(wl.num_seqs, dtype=np.int64)
    step_pairs = []
    for s in range(wl.num_seqs):
        sl, cow = bm.append(s, 1)
        step_slots[s] = sl[0]
        if cow is not None:
            step_pairs.append(cow)
    if pool:
        if step_pairs:
            copy_blocks(kc, vc, np.array(step_pairs))
        reshape_and_cache(kc, vc, kn, vn, step_slots, wl.num_blocks, wl.block_size)
    ctx = np.array([bm.seq_len(s) for s in range(wl.num_seqs)], dtype=np.int64)
    maxb = int(-(-int(ctx.max()) // wl.block_size))
    tables = bm.export_tables(range(wl.num_seqs), maxb)
    res.update({"slots": step_slots, "cow_pairs": np.array(step_pairs, dtype=np.int64).reshape(-1, 2),
                "tables": tables, "ctx_lens": ctx, "q": q, "k_new": kn, "v_new": vn})
    res.pop("out", None)
    if attention and pool:
        res["out"] = paged_attention(q, kc, vc, tables, ctx, wl.scale, wl.dtype, select=select)
    return res
