"""List-based rolling KV cache -- oracle (test infrastructure).

Not for the product path; see the package docstring.

Sources
-------
* "WanToFight: Real-Time Generative Game Engine for Multi-Player Combat
  Interaction", section 三 (技术架构), table "模型组件", rows "Block-Causal
  Attention" and "Rolling KV Cache": inference keeps the KV of the most recent
  2 chunks; older chunks are dropped.  Section "训练流程 / Stage 2" repeats it.
* "Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game
  Worlds", section "前置知识 / 因果自回归与 KV 缓存" and section "技术新颖性":
  the cache keeps the recent-window chunks plus a reference frame, and a ring
  buffer overwrites the oldest slot in place instead of shifting the window.

The logical model is a FIFO list of (chunk id, K, V) records with capacity R:
appending a new chunk pushes it to the back and drops the front when full.
Re-appending the chunk that was appended last replaces it (the clean re-run
of a chunk, "Matrix-Game 4.0", section "方法步骤详情", step 4, and the
penultimate-denoising-step KV of "WanToFight", table "模型组件").

The physical model of the same cache is R slots where chunk ``c`` lives in
slot ``c mod R``; ``expected_physical_slots`` derives it from the list so a test
can compare device memory with it bit for bit.
"""

from __future__ import annotations

from collections import deque

import numpy as np


class RingError(ValueError):
    """A request the rolling cache cannot serve (chunk order, chunk not held)."""


class ListRing:
    """FIFO list of chunk records, capacity ``slots``.

    ``k`` / ``v`` stored per chunk are arrays of any shape (usually
    ``[B, H, Lc, D]``).  The sink (reference chunk) is held separately and is
    never evicted.
    """

    def __init__(self, slots: int):
        if slots < 1:
            raise RingError("ring needs at least one slot")
        self.slots = int(slots)
        self.records: deque = deque()
        self.sink = None  # (k, v) or None

    def set_sink(self, k, v):
        self.sink = (np.array(k, copy=True), np.array(v, copy=True))

    @property
    def last_chunk(self):
        return self.records[-1][0] if self.records else None

    def append(self, chunk: int, k, v):
        chunk = int(chunk)
        last = self.last_chunk
        if last is None:
            if chunk < 0:
                raise RingError("chunk index must be >= 0")
        elif chunk == last:
            self.records.pop()  # rewrite of the newest chunk
        elif chunk != last + 1:
            raise RingError(f"append of chunk {chunk} after chunk {last}: must be {last} or {last + 1}")
        self.records.append((chunk, np.array(k, copy=True), np.array(v, copy=True)))
        while len(self.records) > self.slots:
            self.records.popleft()

    def held_chunks(self) -> list[int]:
        return [r[0] for r in self.records]

    def get(self, chunk: int):
        for c, k, v in self.records:
            if c == chunk:
                return k, v
        raise RingError(f"chunk {chunk} is not held (held: {self.held_chunks()})")


def slot_of(chunk: int, slots: int) -> int:
    """Physical slot of a chunk in an R-slot ring."""
    return int(chunk) % int(slots)


def expected_physical_slots(ring: ListRing, initial: np.ndarray, which: int) -> np.ndarray:
    """Physical contents ``[R, ...]`` implied by the list ring.

    ``initial`` is the ``[R, ...]`` array the slots held before any append
    (slots never written keep it).  ``which`` is 0 for K and 1 for V.  Every
    chunk ever appended overwrote slot ``c mod R``; the chunks still held are
    exactly the last R appended, so replaying the held records in order gives
    the final contents of the slots they occupy.  Slots whose last writer was
    already evicted are not produced by this function: callers compare only
    the slots of held chunks plus slots never written.
    """
    out = np.array(initial, copy=True)
    for c, k, v in ring.records:
        out[slot_of(c, ring.slots)] = k if which == 0 else v
    return out
