"""Reference state machine of the sparse-prefill KV buffer's reuse "head".

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows sglang PR #45909 (SparsePrefillKVBuffer / get_with_head): the buffer
remembers which source it last dequantized -- identified by (source cache,
gather ids, row count), here (layout, pool pointer, pool rows, ids pointer, n)
-- and ``get_with_head`` reports a hit when the same source is asked for
again, so the dequant is skipped.  A plain ``get``, a reallocation, or the
start of a new forward forgets the head.  Skipped dequants are sound because
no later layer of the forward writes the source cache and graph replay keeps
layer order, so a fresh dequant would have written the same rows.
"""
from __future__ import annotations


class KVBufModel:
    def __init__(self, capacity_rows: int):
        if capacity_rows < 0:
            raise ValueError("capacity must be >= 0")
        self.capacity = capacity_rows
        self.head = None
        self.dequants = 0   # number of gather-dequant launches a miss causes

    def realloc(self, capacity_rows: int) -> None:
        if capacity_rows < 0:
            raise ValueError("capacity must be >= 0")
        self.capacity = capacity_rows
        self.head = None

    def begin_forward(self) -> None:
        self.head = None

    def get(self, n: int) -> None:
        if n < 0 or n > self.capacity:
            raise ValueError("n outside [0, capacity]")
        self.head = None

    def get_with_head(self, layout: int, pool: int, pool_rows: int, ids: int,
                      n: int) -> bool:
        """Returns True on a hit (no dequant); on a miss the dequant runs and
        the head becomes this source."""
        if n < 0 or n > self.capacity:
            raise ValueError("n outside [0, capacity]")
        key = (layout, pool, pool_rows, ids, n)
        if self.head == key:
            return True
        self.head = key
        self.dequants += 1
        return False
