"""The seeded input generator: shapes, placement, sharing and the fragmentation bound."""
import numpy as np
import pytest

import workloads as W


def test_tiny_workload_shape_and_pool():
    c = W.make_workload("tiny")
    assert (c.num_seqs, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size) == (4, 4, 4, 64, 16)
    assert c.num_blocks == 64 and c.dtype == "fp16"
    assert c.key_cache.shape == (64, 16, 4, 64) and c.query.shape == (4, 4, 64)
    assert np.all((c.seq_lens >= 1) & (c.seq_lens <= 128))
    assert abs(c.scale - 1 / 8) < 1e-15


def test_deterministic_and_thread_independent():
    a = W.random_case(num_seqs=3, num_q_heads=2, num_kv_heads=1, head_dim=8, block_size=4,
                      len_range=(1, 50), dtype="bf16", seed=7, threads=1)
    b = W.random_case(num_seqs=3, num_q_heads=2, num_kv_heads=1, head_dim=8, block_size=4,
                      len_range=(1, 50), dtype="bf16", seed=7, threads=8)
    for f in ("query", "key_cache", "value_cache", "block_tables", "seq_lens", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    big = W.normal_bits((3, W._CHUNK // 2 + 5), "fp16", 1, 2, threads=1)
    assert np.array_equal(big, W.normal_bits((3, W._CHUNK // 2 + 5), "fp16", 1, 2, threads=4))


def test_random_placement_is_private_and_bounded():
    c = W.random_case(num_seqs=16, num_q_heads=4, num_kv_heads=2, head_dim=8, block_size=8,
                      len_range=(1, 100), dtype="fp16", seed=3)
    B = c.block_size
    used = []
    for s in range(c.num_seqs):
        n = (int(c.seq_lens[s]) + B - 1) // B
        used.extend(c.block_tables[s, :n].tolist())
        # internal fragmentation is at most B - 1 slots per sequence
        assert n * B - int(c.seq_lens[s]) <= B - 1
    assert len(used) == len(set(used))                 # no unintended sharing
    assert c.num_blocks == int(np.ceil(1.2 * len(used)))
    assert np.all((c.block_tables >= 0) & (c.block_tables < c.num_blocks))
    # blocks are not handed out in order
    assert used != sorted(used)


def test_slot_mapping_points_at_last_token():
    c = W.random_case(num_seqs=5, num_q_heads=2, num_kv_heads=2, head_dim=8, block_size=4,
                      len_range=(1, 30), dtype="fp16", seed=2)
    for s in range(5):
        t = int(c.seq_lens[s]) - 1
        assert c.slot_mapping[s] == c.block_tables[s, t // 4] * 4 + t % 4


@pytest.mark.parametrize("B", [1, 4, 16])
def test_shared_prefix_structure(B):
    c = W.shared_prefix_case(block_size=B, groups=3, per_group=4, prefix=16,
                             suffix_range=(0, 10), num_heads=2, head_dim=8, seed=1)
    pre = 16 // B
    for g in range(3):
        rows = c.block_tables[g * 4:(g + 1) * 4, :pre]
        assert np.all(rows == rows[0])                   # one physical prefix per group
    assert not np.array_equal(c.block_tables[0, :pre], c.block_tables[4, :pre])
    assert c.unique_kv_bytes() < c.kv_bytes()
    # sequences without a suffix do not write into the shared prefix
    suf = c.seq_lens - 16
    assert np.all(c.slot_mapping[suf == 0] == -1)


def test_byte_accounting():
    c = W.random_case(num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=8, block_size=4,
                      len_range=(5, 9), dtype="fp16", seed=0, seq_lens=[5, 9])
    kv = 2 * (5 + 9) * 2 * 8 * 2
    assert c.kv_bytes() == kv
    assert c.algorithmic_bytes() == kv + 4 * (2 + 3) + 4 * 2 + 2 * 2 * 4 * 8 * 2
