"""Allocator policy simulator: the oracle.

TEST INFRASTRUCTURE (part of the oracle): only the tests, the smoke check
and the benchmark's CPU legs use it.

Restates the experiment of "The KV Cache Is an Allocator Problem"
(synapticradio.com), section "The experiment": three allocation policies
replay one deterministic trace of requests (arrival step, prompt length,
max_new_tokens, generation length, completion step) against a cache of a
fixed number of token slots:

* max_reservation -- one contiguous interval of prompt + max_new_tokens
  slots, reserved at admission;
* exact_contiguous -- one contiguous interval of prompt slots at admission,
  extended in place one slot per generated token; never relocated;
* paged (block size B) -- blocks of B slots on demand, through the paged
  block manager (pool of floor(capacity / B) blocks, handed out 0, 1, 2, ...).

A request is admitted only if its prompt's cache (for max_reservation, the
whole reservation) can be allocated. At every step the allocator tries to
grow every active request by one token. The recorded quantities are the
section's: admitted and rejected requests, live tokens, reserved slots,
internal waste (reserved minus live), free capacity (capacity minus
reserved), the largest contiguous free interval, and allocation failures
despite sufficient total free capacity; the summary adds the table's growth
failures, peak reserved slots and peak waste.

Readings where the section leaves a step open:
* Step t runs three phases in order: growth of every request admitted
  before t that has generated fewer than its generation length (in trace
  order); completion of every request whose completion step is t (its
  memory is released); admission of every request arriving at t (in trace
  order).
* A failed growth either drops the request (its memory is released and it
  generates no more; the default) or stalls it (it keeps its memory and
  tries again next step).
* Contiguous placement is first fit. Peaks are taken after every successful
  allocation, so they are the instantaneous maxima.
* "Despite sufficient total free capacity": at a failed admission, free
  capacity >= the slots the policy asked for; at a failed growth, free
  capacity >= 1.
* For paged pools the largest contiguous free interval is the longest run of
  free blocks with consecutive ids, times B.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from . import BlockManager
from .contiguous import ContiguousPool

POLICIES = ("max_reservation", "exact_contiguous", "paged")


class _Contiguous:
    def __init__(self, capacity: int, reserve_max: bool):
        self.pool = ContiguousPool(capacity)
        self.capacity = capacity
        self.reserve_max = reserve_max

    def ask(self, req) -> int:
        return req["prompt"] + (req["max_new"] if self.reserve_max else 0)

    def admit(self, rid, req) -> bool:
        return self.pool.reserve(rid, self.ask(req)) is not None

    def grow(self, rid) -> bool:
        if self.reserve_max:
            return True                    # the token was reserved at admission
        return self.pool.grow(rid)

    def release(self, rid):
        self.pool.release(rid)

    def reserved(self) -> int:
        return sum(n for _, n in self.pool.extents.values())

    def largest_free(self) -> int:
        return self.pool.largest_hole()


class _Paged:
    def __init__(self, capacity: int, B: int):
        self.B = B
        self.N = capacity // B
        self.capacity = self.N * B        # slots past the last whole block are unusable
        self.bm = BlockManager(self.N, B, np.arange(self.N, dtype=np.int32))
        self.held: Dict[int, int] = {}

    def ask(self, req) -> int:
        return req["prompt"]

    def admit(self, rid, req) -> bool:
        need = -(-req["prompt"] // self.B)
        if need > self.bm.num_free():
            return False
        self.bm.add_seq(rid)
        self.bm.append(rid, req["prompt"])
        return True

    def grow(self, rid) -> bool:
        try:
            self.bm.append(rid, 1)
        except Exception:
            return False
        return True

    def release(self, rid):
        self.bm.free_seq(rid)

    def reserved(self) -> int:
        return (self.N - self.bm.num_free()) * self.B

    def largest_free(self) -> int:
        free = sorted(int(b) for b in self.bm.free_list())
        best = run = 0
        prev = None
        for b in free:
            run = run + 1 if prev is not None and b == prev + 1 else 1
            best = max(best, run)
            prev = b
        return best * self.B


def simulate(trace: List[dict], capacity: int, policy: str, block_size: int = 0,
             on_growth_failure: str = "drop") -> dict:
    """Replays ``trace`` (dicts with arrival, prompt, max_new, gen, completion)
    under one policy. Returns the summary counters and one sample per step
    (taken at the end of the step)."""
    if policy == "paged":
        alloc = _Paged(capacity, block_size)
    elif policy in ("max_reservation", "exact_contiguous"):
        alloc = _Contiguous(capacity, policy == "max_reservation")
    else:
        raise ValueError(policy)
    drop = on_growth_failure == "drop"
    n = len(trace)
    state = ["waiting"] * n          # waiting, active, rejected, dropped, done
    generated = [0] * n
    admitted_at = [-1] * n
    c = dict(admitted=0, rejected=0, rejected_despite_free=0, growth_failures=0,
             growth_failures_despite_free=0, dropped=0, completed=0,
             peak_live=0, peak_reserved=0, peak_waste=0)

    def live() -> int:
        return sum(trace[i]["prompt"] + generated[i] for i in range(n) if state[i] == "active")

    def note_peaks():
        lv, rs = live(), alloc.reserved()
        c["peak_live"] = max(c["peak_live"], lv)
        c["peak_reserved"] = max(c["peak_reserved"], rs)
        c["peak_waste"] = max(c["peak_waste"], rs - lv)

    last = max([r["completion"] for r in trace] + [r["arrival"] for r in trace] + [0])
    samples = []
    for t in range(last + 1):
        # growth
        for i in range(n):
            if state[i] != "active" or admitted_at[i] >= t or generated[i] >= trace[i]["gen"]:
                continue
            if alloc.grow(i):
                generated[i] += 1
                note_peaks()
                continue
            c["growth_failures"] += 1
            if alloc.capacity - alloc.reserved() >= 1:
                c["growth_failures_despite_free"] += 1
            if drop:
                alloc.release(i)
                state[i] = "dropped"
                c["dropped"] += 1
        # completion
        for i in range(n):
            if state[i] == "active" and trace[i]["completion"] == t:
                alloc.release(i)
                state[i] = "done"
                c["completed"] += 1
        # admission
        for i in range(n):
            if state[i] != "waiting" or trace[i]["arrival"] != t:
                continue
            free_before = alloc.capacity - alloc.reserved()
            if alloc.admit(i, trace[i]):
                state[i] = "active"
                admitted_at[i] = t
                c["admitted"] += 1
                note_peaks()
            else:
                state[i] = "rejected"
                c["rejected"] += 1
                if free_before >= alloc.ask(trace[i]):
                    c["rejected_despite_free"] += 1
        lv, rs = live(), alloc.reserved()
        samples.append(dict(step=t, active=sum(s == "active" for s in state), live=lv, reserved=rs,
                            waste=rs - lv, free=alloc.capacity - rs, largest_free=alloc.largest_free()))
    return {"summary": c, "samples": samples}
