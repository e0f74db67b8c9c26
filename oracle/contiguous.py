"""Contiguous first-fit reservation: the allocator that paging replaces.

TEST INFRASTRUCTURE (part of the oracle). It exists only to pin the pages'
contrast between contiguous placement and paged placement:

* "The KV Cache Is an Allocator Problem" (synapticradio.com), section "One
  request, two kinds of waste": an 80-slot cache in which a request fails to
  find one contiguous interval although enough slots are free in total.
* "Paged KV Cache Allocation and the Block Table" (mercemay.com), section
  "Three ways contiguous reservation loses memory": external fragmentation.

Each request reserves one interval [start, start + n); placement is first fit
(the lowest free start that fits). An interval grows in place by one slot when
the slot after it is free. Freeing returns the interval.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple


class ContiguousPool:
    def __init__(self, num_slots: int):
        self.num_slots = int(num_slots)
        self.extents: Dict[int, Tuple[int, int]] = {}  # request id -> (start, length)

    def holes(self) -> List[Tuple[int, int]]:
        """Free intervals as (start, length), in address order."""
        taken = sorted(self.extents.values())
        out, pos = [], 0
        for start, n in taken:
            if start > pos:
                out.append((pos, start - pos))
            pos = max(pos, start + n)
        if pos < self.num_slots:
            out.append((pos, self.num_slots - pos))
        return out

    def free_slots(self) -> int:
        return sum(n for _, n in self.holes())

    def largest_hole(self) -> int:
        return max((n for _, n in self.holes()), default=0)

    def reserve(self, rid: int, n: int) -> Optional[int]:
        """First-fit placement of n contiguous slots; None if no hole fits."""
        for start, length in self.holes():
            if length >= n:
                self.extents[rid] = (start, n)
                return start
        return None

    def grow(self, rid: int) -> bool:
        """Extends the request's interval by one slot in place (no
        relocation): succeeds only if the slot right after it is free."""
        start, n = self.extents[rid]
        end = start + n
        if end >= self.num_slots:
            return False
        for other, (s2, n2) in self.extents.items():
            if other != rid and s2 <= end < s2 + n2:
                return False
        self.extents[rid] = (start, n + 1)
        return True

    def release(self, rid: int):
        del self.extents[rid]
