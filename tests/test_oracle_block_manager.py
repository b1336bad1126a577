"""Pins for the CPU block-manager model (oracle/block_manager.py).

* the copy-on-write example printed in "PagedAttention by hand" (Why divide
  memory into physical blocks?, Example of Copy-on-Write): a 5-token prompt in
  blocks of 2 shared by two candidates; the first candidate to write token 6
  copies only the last block, the second writes in place, the first two blocks
  stay shared with a reference count of 2;
* the glossary's rule that a sequence gets a new physical block only once its
  previous block is full, and the by-hand page's waste bound of at most B - 1
  slots per sequence;
* invariants recomputed from the tables by brute force: reference counts equal
  the number of tables holding a block, free + used blocks = pool size.
"""
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManager, CapacityError, copy_blocks


def _check_invariants(bm):
    count = [0] * bm.num_blocks
    for t in bm.tables.values():
        assert len(set(t)) == len(t)
        for b in t:
            count[b] += 1
    assert count == bm.ref
    used = {b for t in bm.tables.values() for b in t}
    assert len(used) + len(bm.free) == bm.num_blocks
    assert used.isdisjoint(bm.free)
    for sid, t in bm.tables.items():
        L = bm.lens[sid]
        assert len(t) == (L + bm.B - 1) // bm.B
        assert len(t) * bm.B - L <= bm.B - 1  # internal fragmentation bound


def test_copy_on_write_example_from_the_page():
    bm = BlockManager(num_blocks=9, block_size=2, max_blocks_per_seq=8)
    a = bm.new_sequence()
    slots, copies = bm.append([(a, 5)])  # prompt t1..t5 in [t1,t2] [t3,t4] [t5,_]
    assert copies == [] and len(bm.tables[a]) == 3
    b = bm.fork(a)                       # candidate B shares the mapping
    shared = list(bm.tables[a])
    assert bm.tables[b] == shared and all(bm.ref[x] == 2 for x in shared)
    # candidate A writes token 6 into slot 1 of logical block 2 (refcount 2)
    slots_a, copies_a = bm.append([(a, 1)])
    assert len(copies_a) == 1 and copies_a[0][0] == shared[2]
    new = copies_a[0][1]
    assert new not in shared
    assert bm.tables[a] == shared[:2] + [new]
    assert slots_a == [new * 2 + 1]
    assert bm.ref[shared[2]] == 1 and bm.ref[new] == 1
    # candidate B: refcount is now 1 -> writes k6/v6 directly into the old block
    slots_b, copies_b = bm.append([(b, 1)])
    assert copies_b == [] and slots_b == [shared[2] * 2 + 1]
    # blocks holding t1-t4 are still shared with reference count 2
    assert bm.ref[shared[0]] == 2 and bm.ref[shared[1]] == 2
    _check_invariants(bm)


def test_both_candidates_in_one_append_copy_once():
    bm = BlockManager(9, 2, 8)
    a = bm.new_sequence()
    bm.append([(a, 5)])
    b = bm.fork(a)
    slots, copies = bm.append([(a, 1), (b, 1)])
    assert len(copies) == 1
    assert slots[1] == bm.tables[b][2] * 2 + 1 and slots[0] == bm.tables[a][2] * 2 + 1
    _check_invariants(bm)


def test_blocks_allocated_only_when_the_previous_fills():
    B = 4
    bm = BlockManager(20, B, 10)
    s = bm.new_sequence()
    for t in range(23):
        before = len(bm.tables[s])
        slots, _ = bm.append([(s, 1)])
        after = len(bm.tables[s])
        assert after - before == (1 if t % B == 0 else 0)
        assert slots == [bm.tables[s][t // B] * B + t % B]
    _check_invariants(bm)


def test_fresh_pool_hands_out_block_ids_in_order_and_reuses_freed_ones_last_in_first_out():
    bm = BlockManager(8, 4, 8)
    s = bm.new_sequence()
    bm.append([(s, 9)])
    assert bm.tables[s] == [0, 1, 2]
    bm.free_sequence(s)
    t = bm.new_sequence()
    bm.append([(t, 1)])
    assert bm.tables[t] == [2]  # the last block pushed is on top


def test_capacity_errors_leave_the_state_unchanged():
    bm = BlockManager(3, 2, 8)
    s = bm.new_sequence()
    bm.append([(s, 4)])
    snapshot = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lens))
    with pytest.raises(CapacityError):
        bm.append([(s, 3)])  # needs 2 more blocks, 1 free
    assert snapshot == (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lens))
    small = BlockManager(16, 2, 2)
    q = small.new_sequence()
    with pytest.raises(CapacityError):
        small.append([(q, 5)])  # table holds 2 blocks = 4 tokens


def test_random_operations_keep_the_invariants():
    rng = random.Random(5)
    bm = BlockManager(64, 4, 32)
    live = []
    for _ in range(600):
        op = rng.random()
        try:
            if op < 0.15 or not live:
                live.append(bm.new_sequence())
            elif op < 0.3:
                live.append(bm.fork(rng.choice(live)))
            elif op < 0.4 and len(live) > 1:
                sid = live.pop(rng.randrange(len(live)))
                bm.free_sequence(sid)
            else:
                k = rng.randint(1, min(4, len(live)))
                reqs = [(sid, rng.randint(1, 6)) for sid in rng.sample(live, k)]
                bm.append(reqs)
        except CapacityError:
            pass
        _check_invariants(bm)


def test_copy_blocks_moves_whole_blocks():
    kc = np.arange(5 * 2 * 3, dtype=np.uint16).reshape(5, 2, 3)
    vc = kc + 100
    k0, v0 = kc.copy(), vc.copy()
    copy_blocks(kc, vc, [(1, 3), (4, 0)])
    assert np.array_equal(kc[3], k0[1]) and np.array_equal(vc[3], v0[1])
    assert np.array_equal(kc[0], k0[4]) and np.array_equal(vc[0], v0[4])
    for b in (1, 2, 4):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
