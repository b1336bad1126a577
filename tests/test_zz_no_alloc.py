"""pa_decode_no_alloc: the decode entry point for callers that cannot allocate
device memory (its split-K scratch is a fixed array inside the library).

It must give the same output as pa_decode with a caller-owned workspace, call
after call, although every call reuses the same scratch. This file is named
to be collected last, so a run that stops at the first failure has already run
every other test.
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


def _no_alloc(dc, out, pt):
    return pa.decode_no_alloc(out, dc.query, dc.key_cache, dc.value_cache, dc.block_tables,
                              dc.seq_lens, dc.case.scale, pt)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_no_alloc_matches_workspace_decode_on_two_calls(dtype):
    # several partitions per sequence, so the scratch (partials + counters) is used
    case = W.random_case(num_seqs=6, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                         len_range=(1, 3000), dtype=dtype, seed=21, partition_tokens=128)
    dc = DeviceCase(case)
    want16 = host_bits(dc.decode()).copy()
    want32 = dc.decode(out_f32=True).cpu().numpy().copy()
    ref = oracle.paged_decode(case.query, case.key_cache, case.value_cache, case.block_tables,
                              case.seq_lens, case.block_size, case.scale, dtype)
    for call in range(2):
        out16 = torch.full(dc.query.shape, float("nan"), dtype=dc.query.dtype, device="cuda")
        out32 = torch.full(dc.query.shape, float("nan"), dtype=torch.float32, device="cuda")
        _no_alloc(dc, out16, 128)
        _no_alloc(dc, out32, 128)
        torch.cuda.synchronize()
        # the same kernel and schedule as pa_decode: the same bits
        assert np.array_equal(host_bits(out16), want16), call
        assert np.array_equal(out32.cpu().numpy(), want32), call
        check_parity(host_bits(out16), out32.cpu().numpy(), ref, dtype, f"no-alloc call {call}")


def test_no_alloc_after_a_different_shape():
    # The scratch keeps the previous call's contents. The small call (2 x 32
    # query heads = 64 rows) leaves its fp32 log-sum-exp values right after
    # its 64 counters; the big call's 40 x 8 counters then cover those bytes.
    # Every row of both is cut into pieces, so every row goes through a counter.
    small = W.random_case(num_seqs=2, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          len_range=(2500, 3000), dtype="bf16", seed=22, partition_tokens=16)
    big = W.random_case(num_seqs=40, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                        len_range=(2500, 3000), dtype="bf16", seed=23, partition_tokens=64)
    for case in (big, small, big):
        dc = DeviceCase(case)
        # pa_decode on a freshly zeroed workspace of its own
        want = dc.decode(out_f32=True).cpu().numpy().copy()
        out = torch.full(dc.query.shape, float("nan"), dtype=torch.float32, device="cuda")
        _no_alloc(dc, out, case.partition_tokens)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want), case.num_seqs


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    limit = pa.no_alloc_scratch_bytes()
    assert limit == 64 << 20
    case = W.random_case(num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                         len_range=(1, 64), dtype="fp16", seed=24)
    dc = DeviceCase(case)
    # a table wide enough that the split-K scratch would exceed the limit
    wide = torch.zeros((2, 1 << 20), dtype=torch.int32, device="cuda")
    need = pa.decode_workspace_bytes(2, 4, 64, wide.shape[1], 16, 16)
    assert need > limit
    with pytest.raises(pa.PagedAttnError, match="scratch"):
        pa.decode_no_alloc(dc.out, dc.query, dc.key_cache, dc.value_cache, wide, dc.seq_lens,
                           case.scale, 16)
