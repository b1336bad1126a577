"""The library's native block manager (host code, no GPU needed) against the
CPU model in oracle/block_manager.py: identical slots, copy-on-write copies,
tables, lengths, reference counts and free counts over random operation
sequences, and the same capacity errors."""
import random

import numpy as np
import pytest

import paged_kv_cache_305_gb300 as pa
from oracle.block_manager import BlockManager as Model, CapacityError
from paged_kv_cache_305_gb300 import build as pbuild


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    pa.load_library()


def _same_state(bm, model, live):
    assert bm.num_free_blocks() == len(model.free)
    for b in range(model.num_blocks):
        assert bm.ref_count(b) == model.ref[b]
    if live:
        tables, lens = bm.block_tables(live)
        mt, ml = model.table_rows(live)
        assert np.array_equal(tables, np.array(mt, dtype=np.int32))
        assert lens.tolist() == ml


@pytest.mark.parametrize("seed,B,NB,MB", [(0, 2, 9, 8), (1, 16, 64, 16), (2, 1, 40, 64), (3, 4, 30, 10)])
def test_native_manager_matches_the_model(seed, B, NB, MB):
    rng = random.Random(seed)
    bm = pa.BlockManager(NB, B, MB)
    model = Model(NB, B, MB)
    live = []
    for _ in range(400):
        op = rng.random()
        if op < 0.15 or not live:
            a, b = bm.new_sequence(), model.new_sequence()
            assert a == b
            live.append(a)
        elif op < 0.3:
            p = rng.choice(live)
            a, b = bm.fork(p), model.fork(p)
            assert a == b
            live.append(a)
        elif op < 0.4 and len(live) > 1:
            sid = live.pop(rng.randrange(len(live)))
            bm.free_sequence(sid)
            model.free_sequence(sid)
        else:
            k = rng.randint(1, min(5, len(live)))
            reqs = [(sid, rng.randint(0, 2 * B + 1)) for sid in rng.sample(live, k)]
            try:
                want = model.append(reqs)
            except CapacityError:
                with pytest.raises(pa.PagedAttnError) as e:
                    bm.append(reqs)
                assert e.value.code == pa.PA_ERR_CAPACITY
            else:
                slots, copies = bm.append(reqs)
                assert slots.tolist() == want[0]
                assert copies == want[1]
        _same_state(bm, model, live)


def test_copy_on_write_example_on_the_native_manager():
    # "PagedAttention by hand": 5-token prompt, blocks of 2, two candidates
    bm = pa.BlockManager(9, 2, 8)
    a = bm.new_sequence()
    slots, copies = bm.append([(a, 5)])
    assert slots.tolist() == [0, 1, 2, 3, 4] and copies == []
    b = bm.fork(a)
    assert [bm.ref_count(x) for x in (0, 1, 2)] == [2, 2, 2]
    slots, copies = bm.append([(a, 1), (b, 1)])
    assert copies == [(2, 3)]           # only A's last block is duplicated
    assert slots.tolist() == [3 * 2 + 1, 2 * 2 + 1]
    assert [bm.ref_count(x) for x in (0, 1, 2, 3)] == [2, 2, 1, 1]


@pytest.mark.parametrize("call", ["bad_seq", "dup", "neg", "free_twice", "fork_dead"])
def test_native_manager_rejects_bad_calls(call):
    bm = pa.BlockManager(8, 4, 4)
    a = bm.new_sequence()
    with pytest.raises(pa.PagedAttnError) as e:
        if call == "bad_seq":
            bm.append([(a + 7, 1)])
        elif call == "dup":
            bm.append([(a, 1), (a, 2)])
        elif call == "neg":
            bm.append([(a, -1)])
        elif call == "free_twice":
            bm.free_sequence(a)
            bm.free_sequence(a)
        else:
            bm.free_sequence(a)
            bm.fork(a)
    assert e.value.code == -1


def test_capacity_error_changes_nothing():
    bm = pa.BlockManager(3, 2, 8)
    a = bm.new_sequence()
    bm.append([(a, 4)])
    before = (bm.num_free_blocks(), bm.block_tables([a]))
    with pytest.raises(pa.PagedAttnError) as e:
        bm.append([(a, 3)])
    assert e.value.code == pa.PA_ERR_CAPACITY
    after = (bm.num_free_blocks(), bm.block_tables([a]))
    assert before[0] == after[0] and np.array_equal(before[1][0], after[1][0])
    small = pa.BlockManager(16, 2, 2)
    q = small.new_sequence()
    with pytest.raises(pa.PagedAttnError) as e:
        small.append([(q, 5)])
    assert e.value.code == pa.PA_ERR_CAPACITY


def test_create_rejects_bad_sizes():
    with pytest.raises(pa.PagedAttnError):
        pa.BlockManager(0, 16, 4)
