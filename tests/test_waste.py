"""KV-memory waste: the accounting oracle pinned to the numbers printed on the
pages, and the simulator (driving the library's native block manager)
checked step by step against that accounting."""
import pytest

from oracle.waste import contiguous_waste, paged_waste
from paged_kv_cache_305_gb300 import build as pbuild


def test_page_examples_of_contiguous_reservation():
    # "PagedAttention by hand", Why divide memory into physical blocks?, 1.:
    # max length 2048, a 50-token prompt wastes 1998 slots; after a 10-token
    # answer 1988 slots are still wasted
    assert contiguous_waste([50], 2048) == (1998, 2048)
    assert contiguous_waste([60], 2048) == (1988, 2048)


def test_page_example_of_paged_allocation():
    # the by-hand page: 5 tokens in blocks of 2 take 3 blocks (6 slots), one slot unused
    assert paged_waste([5], 2) == (1, 6)


def test_paged_waste_is_at_most_block_size_minus_one_per_sequence():
    for B in (1, 2, 8, 16, 64):
        worst = max(paged_waste([L], B)[0] for L in range(1, 3 * B + 5))
        assert worst == B - 1
    # the by-hand page: about 15 wasted slots per sequence at B = 16, whatever
    # the length (here 20 or 20000 tokens)
    assert paged_waste([20], 16)[0] <= 15 and paged_waste([20000], 16)[0] <= 15
    assert max(paged_waste([20000 + k], 16)[0] for k in range(16)) == 15


@pytest.mark.parametrize("B", [1, 16, 64])
def test_simulator_matches_the_accounting_step_by_step(B):
    pbuild.build()
    from paged_kv_cache_305_gb300 import waste
    trace = []
    r = waste.simulate(block_size=B, concurrent=16, requests=64, seed=B, trace=trace)
    used = sum(sum(t) for t in trace)
    paged = sum(paged_waste(t, B)[1] for t in trace)
    contig = sum(contiguous_waste(t, r.max_len)[1] for t in trace)
    assert (used, paged, contig) == (r.used_token_steps, r.paged_slot_steps, r.contiguous_slot_steps)
    assert r.max_paged_waste_per_seq <= B - 1
