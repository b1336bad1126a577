"""Full-size workloads on the GPU, in the launch configuration bench.py times.

Every (sequence, query head) output row of every workload is compared with
the float64 oracle (fp32 result within 2e-3, 16-bit output its nearest-even
rounding). The step: write each sequence's newest token with
pa_reshape_and_cache, then pa_decode over the whole sequence; and, where
every newest token has a block of its own, the fused pa_decode_append that
the benchmark times by default, which must give the same bits.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import paged_kv_cache_305_gb300 as pa
import workloads as W
from gpu_util import DeviceCase, check_parity, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_305_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _run_and_check(case):
    dc = DeviceCase(case)
    out = dc.step()
    torch.cuda.synchronize()
    got = host_bits(out).copy()
    got32 = dc.decode(out_f32=True).cpu().numpy()
    if np.all(case.slot_mapping >= 0):
        # the fused step bench.py times by default: the same bits (its new rows
        # are the ones the separate write stored, so the caches do not change)
        fused = torch.empty_like(dc.query)
        pa.decode_append(fused, dc.query, dc.new_key, dc.new_value, dc.key_cache, dc.value_cache,
                         dc.block_tables, dc.seq_lens, case.scale, dc.partition_tokens, dc.workspace)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(fused), got)
    # every 16-bit output is the nearest-even rounding of the fp32 result
    assert np.array_equal(oracle.round_to_dtype(got32.astype(np.float64), case.dtype), got)
    # the written rows are where the oracle's write puts them
    B = case.block_size
    for s in range(case.num_seqs):
        sl = int(case.slot_mapping[s])
        if sl >= 0:
            assert np.array_equal(host_bits(dc.key_cache[sl // B, sl % B]), case.new_key[s])
            assert np.array_equal(host_bits(dc.value_cache[sl // B, sl % B]), case.new_value[s])
    kc, vc = oracle.reshape_and_cache(case.new_key, case.new_value, case.key_cache,
                                      case.value_cache, case.slot_mapping, B, in_place=True)
    del dc
    torch.cuda.empty_cache()
    # the oracle over the whole batch: every row, every head
    ref = oracle.paged_decode(case.query, kc, vc, case.block_tables, case.seq_lens, B,
                              case.scale, case.dtype)
    err = check_parity(got, got32, ref, case.dtype,
                       f"{case.name} (all {case.num_seqs * case.num_q_heads} rows)")
    return err


@pytest.mark.parametrize("name", ["llama2_7b_mha", "llama3_8b_gqa", "long_context_splitk"])
def test_full_size_workload(name):
    _run_and_check(W.make_workload(name))


@pytest.mark.parametrize("B", W.SHARED_PREFIX_BLOCK_SIZES)
def test_shared_prefix_block_size_sweep(B):
    _run_and_check(W.make_workload("shared_prefix", block_size=B))
