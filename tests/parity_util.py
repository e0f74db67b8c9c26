"""Shared pieces of the GPU parity tests: error metrics and the tolerances.

Tolerances (element by element against the double-precision oracle):
* bf16 attention: max-abs <= 1e-2 and relative L2 <= 2e-3 (the stated bar).
* fp32 attention: max-abs <= 1e-5 and relative L2 <= 2e-6. Derivation: the
  kernel accumulates in fp32 (unit roundoff 6e-8); a score carries about
  sqrt(d) * 6e-8 relative error and exp2f at most 2 ulp, so each softmax
  weight is off by ~1e-6 relative at worst, and outputs (weighted means of
  N(0,1) values, |out| < 4) by a few 1e-7 typically and ~1e-6 at worst.
* Scatter, block tables, slot mappings and block copies: bit-exact.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from workloads import bf16_bits_to_f32

TOL = {"bf16": (1e-2, 2e-3), "f32": (1e-5, 2e-6)}


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return a.astype(np.float64) if dtype == "f32" else bf16_bits_to_f32(a).astype(np.float64)


def errors(got: np.ndarray, want: np.ndarray):
    d = got - want
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(want), 1e-300))


def assert_close(got_bits: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    got = as_f64(got_bits, dtype)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx, rl = errors(got, want)
    tmax, trel = TOL[dtype]
    assert mx <= tmax and rl <= trel, f"{what}: max-abs {mx:.3g} (<= {tmax}), rel-L2 {rl:.3g} (<= {trel})"
    return mx, rl


_POOL = None


def _host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_every_row(ref: dict, wl) -> np.ndarray:
    """The oracle's attention for every (sequence, query head) row of the
    step held in ``ref`` (an ``oracle.run_workload`` / ``continue_workload``
    result), float64 ``[S, Hq, d]``.

    The rows are dealt longest context first, round-robin, to one host thread
    per core; each thread calls the (reentrant, single-threaded) C oracle on
    its share, and ctypes releases the interpreter lock for the call. Each
    row is computed exactly as a single call over all rows would compute it.
    """
    import oracle
    global _POOL
    S, Hq = wl.num_seqs, wl.num_q_heads
    rows = np.array([(s, h) for s in range(S) for h in range(Hq)], dtype=np.int32)
    ctx = np.asarray(ref["ctx_lens"])
    threads = max(1, min(_host_threads(), len(rows) // 4))
    order = np.argsort(-ctx[rows[:, 0]], kind="stable")
    shares = [np.ascontiguousarray(rows[order[i::threads]]) for i in range(threads)]
    args = (ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"], wl.scale, wl.dtype)
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=_host_threads())
    parts = list(_POOL.map(lambda sel: (sel, oracle.paged_attention(*args, select=sel)), shares))
    out = np.full((S, Hq, wl.head_dim), np.nan, dtype=np.float64)
    for sel, part in parts:
        out[sel[:, 0], sel[:, 1]] = part[sel[:, 0], sel[:, 1]]
    assert np.isfinite(out).all(), "the oracle left a row uncomputed"
    return out
