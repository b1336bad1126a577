"""KV-memory waste accounting -- TEST INFRASTRUCTURE ONLY (see oracle/__init__).

Written from "PagedAttention by hand" (What is PagedAttention: the waste
table; Why divide memory into physical blocks?, 1. Zero External
Fragmentation) and the "PagedAttention" glossary (Why It Exists):

* contiguous pre-reservation holds `max_len` slots per request from admission,
  so a request that has `used` tokens wastes max_len - used slots (reserved +
  internal fragmentation);
* paging allocates on demand in blocks of B, so it wastes only the empty
  tail of the last block: ceil(used / B) * B - used, at most B - 1.
"""
from __future__ import annotations

from typing import Iterable


def contiguous_waste(used: Iterable[int], max_len: int):
    """(wasted slots, reserved slots) under max_len pre-reservation."""
    used = list(used)
    reserved = max_len * len(used)
    return reserved - sum(used), reserved


def paged_waste(used: Iterable[int], block_size: int):
    """(wasted slots, allocated slots) with on-demand blocks of block_size."""
    B = block_size
    alloc = sum((u + B - 1) // B * B for u in used)
    return alloc - sum(used), alloc
