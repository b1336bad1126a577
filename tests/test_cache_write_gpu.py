"""GPU parity of pa_reshape_and_cache (through the C ABI): bit-exact against
the oracle's element copy, for both 16-bit types and both head sizes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import paged_kv_cache_305_gb300 as pa
import workloads as W
from gpu_util import DeviceCase, dev_bits, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_305_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype,Hkv,d,B", [("fp16", 4, 64, 16), ("bf16", 8, 128, 16),
                                           ("bf16", 1, 64, 1), ("fp16", 3, 128, 64)])
def test_random_slots_bit_exact(dtype, Hkv, d, B):
    case = W.random_case(num_seqs=3, num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=(1, 200), dtype=dtype, seed=Hkv + d)
    T = 97
    rng = np.random.default_rng(0)
    key = W.normal_bits((T, Hkv, d), dtype, 5, 1)
    val = W.normal_bits((T, Hkv, d), dtype, 5, 2)
    slots = rng.choice(case.num_blocks * B, size=T, replace=False).astype(np.int64)
    slots[::7] = -1
    kc_d, vc_d = dev_bits(case.key_cache, dtype), dev_bits(case.value_cache, dtype)
    pa.reshape_and_cache(dev_bits(key, dtype), dev_bits(val, dtype), kc_d, vc_d,
                         torch.from_numpy(slots).cuda())
    kc, vc = oracle.reshape_and_cache(key, val, case.key_cache, case.value_cache, slots, B)
    assert np.array_equal(host_bits(kc_d), kc)
    assert np.array_equal(host_bits(vc_d), vc)


def test_fill_whole_sequences_through_the_table():
    # a prefill-sized write: every token of every sequence, addressed by slot
    case = W.random_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                         len_range=(1, 500), dtype="bf16", seed=11)
    B = case.block_size
    slots, rows = [], []
    for s in range(case.num_seqs):
        for t in range(int(case.seq_lens[s])):
            slots.append(int(case.block_tables[s, t // B]) * B + t % B)
    T = len(slots)
    key = W.normal_bits((T, 2, 128), "bf16", 9, 1)
    val = W.normal_bits((T, 2, 128), "bf16", 9, 2)
    zero = np.zeros_like(case.key_cache)
    kc_d, vc_d = dev_bits(zero, "bf16"), dev_bits(zero, "bf16")
    sl = np.array(slots, np.int64)
    pa.reshape_and_cache(dev_bits(key, "bf16"), dev_bits(val, "bf16"), kc_d, vc_d,
                         torch.from_numpy(sl).cuda())
    kc, vc = oracle.reshape_and_cache(key, val, zero, zero, sl, B)
    assert np.array_equal(host_bits(kc_d), kc) and np.array_equal(host_bits(vc_d), vc)
    # reading back through the table returns the rows in logical order
    K = oracle.gather_kv(host_bits(kc_d), case.block_tables[0], int(case.seq_lens[0]), B)
    assert np.array_equal(K, key[: int(case.seq_lens[0])])


def test_out_of_range_slot_is_skipped_and_counted():
    case = W.make_workload("tiny")
    dc = DeviceCase(case)
    before = host_bits(dc.key_cache).copy()
    pa.bad_index_count(clear=True)
    bad = torch.tensor([case.num_blocks * case.block_size, -1, 10 ** 12, -5], dtype=torch.int64,
                       device="cuda")
    pa.reshape_and_cache(dc.new_key[:4], dc.new_value[:4], dc.key_cache, dc.value_cache, bad)
    assert pa.bad_index_count(clear=True) == 2
    assert np.array_equal(host_bits(dc.key_cache), before)


def test_decode_step_write_lands_where_decode_reads():
    case = W.make_workload("tiny")
    dc = DeviceCase(case)
    dc.write_new_tokens()
    kc, vc = oracle.reshape_and_cache(case.new_key, case.new_value, case.key_cache,
                                      case.value_cache, case.slot_mapping, case.block_size)
    assert np.array_equal(host_bits(dc.key_cache), kc)
    assert np.array_equal(host_bits(dc.value_cache), vc)
