"""Plain CPU model of the paged KV-cache block manager -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and ``bench.py`` may import this module; the library's native
block manager (``csrc/block_manager.cpp``) shares no code with it.

What it models ("PagedAttention by hand", What is PagedAttention and Why
divide memory into physical blocks?; the "PagedAttention" glossary, How It
Works):

* The pool is ``num_blocks`` fixed-size blocks of ``block_size`` token slots.
  Free blocks sit on a stack of interchangeable ids.
* A sequence owns a block table; a new physical block is taken only when the
  previous one is full (token t goes to logical block t // B, offset t % B).
* Forking a sequence (e.g. sampling n = 2 candidates from one prompt) shares
  every block of the parent: each shared block's reference count goes up.
* Writing a token into a block whose reference count is above 1 is a
  copy-on-write: take a fresh block, copy that one block, decrement the old
  block's count, and write into the copy. A candidate that later writes into
  a block whose count has dropped back to 1 writes in place.
* Freeing a sequence decrements its blocks' counts; blocks reaching 0 go back
  on the free stack.

The pages fix no order for the free stack; this model (and the library) use
one definite policy so results can be compared exactly: the stack starts as
[num_blocks-1, ..., 1, 0] (block 0 on top, so a fresh pool hands out 0, 1,
2, ...), a freed sequence pushes its blocks in table order, and allocation
pops the top.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


class CapacityError(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self.B = block_size
        self.num_blocks = num_blocks
        self.max_blocks_per_seq = max_blocks_per_seq
        self.free: List[int] = list(range(num_blocks - 1, -1, -1))  # top = end
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self._next_id = 0
        self._free_ids: List[int] = []

    # -- sequences -----------------------------------------------------------
    def new_sequence(self) -> int:
        sid = self._free_ids.pop() if self._free_ids else self._take_id()
        self.tables[sid] = []
        self.lens[sid] = 0
        return sid

    def _take_id(self) -> int:
        sid = self._next_id
        self._next_id += 1
        return sid

    def fork(self, parent: int) -> int:
        """A child that shares every block of ``parent`` (reference counts + 1)."""
        child = self.new_sequence()
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1
        return child

    def free_sequence(self, sid: int) -> None:
        for b in self.tables.pop(sid):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[sid]
        self._free_ids.append(sid)

    # -- appending tokens ----------------------------------------------------
    def _blocks_needed(self, requests: Sequence[Tuple[int, int]]) -> int:
        """Blocks an append of these (sequence, count) requests takes, in order."""
        need = 0
        extra_refs: Dict[int, int] = {}
        for sid, n in requests:
            L = self.lens[sid]
            for t in range(L, L + n):
                off = t % self.B
                if off == 0:
                    need += 1
                elif t == L:
                    blk = self.tables[sid][t // self.B]
                    if self.ref[blk] + extra_refs.get(blk, 0) > 1:
                        need += 1
                        extra_refs[blk] = extra_refs.get(blk, 0) - 1
        return need

    def append(self, requests: Sequence[Tuple[int, int]]):
        """Reserve slots for ``n`` new tokens of each listed sequence, in order.

        Returns (slots, copies): one slot (block * B + offset) per new token,
        in request order, and the (source, destination) block copies that
        copy-on-write needs before the new tokens are written. Raises
        CapacityError (with nothing changed) if the pool or a table is too small.
        """
        seen = set()
        for sid, n in requests:
            if sid in seen:
                raise ValueError("a sequence may appear once per append")
            seen.add(sid)
            if (self.lens[sid] + n + self.B - 1) // self.B > self.max_blocks_per_seq:
                raise CapacityError("block table full")
        if self._blocks_needed(requests) > len(self.free):
            raise CapacityError("out of blocks")
        slots: List[int] = []
        copies: List[Tuple[int, int]] = []
        for sid, n in requests:
            table = self.tables[sid]
            for _ in range(n):
                t = self.lens[sid]
                lb, off = divmod(t, self.B)
                if off == 0:
                    blk = self.free.pop()
                    self.ref[blk] = 1
                    table.append(blk)
                else:
                    blk = table[lb]
                    if self.ref[blk] > 1:  # copy-on-write
                        new = self.free.pop()
                        self.ref[new] = 1
                        self.ref[blk] -= 1
                        copies.append((blk, new))
                        table[lb] = new
                        blk = new
                slots.append(blk * self.B + off)
                self.lens[sid] = t + 1
        return slots, copies

    # -- export --------------------------------------------------------------
    def table_rows(self, sids: Sequence[int]):
        """(tables [len(sids), max_blocks_per_seq] padded with 0, lengths)."""
        rows = []
        for sid in sids:
            t = self.tables[sid]
            rows.append(t + [0] * (self.max_blocks_per_seq - len(t)))
        return rows, [self.lens[s] for s in sids]


def copy_blocks(key_cache: np.ndarray, value_cache: np.ndarray, pairs) -> None:
    """Copy-on-write's device step: block src's contents onto block dst, in both
    caches, for each (src, dst) pair, in place."""
    for src, dst in pairs:
        key_cache[dst] = key_cache[src]
        value_cache[dst] = value_cache[src]
