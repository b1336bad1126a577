"""GPU parity of pa_decode (through the C ABI) against the float64 CPU oracle.

Small cases that the oracle finishes in seconds but that still span several
16-token tiles, several warps' token rounds and several split-K partitions,
with ragged tails, plus the method's degenerate cases. Tolerance: max |err|
<= 2e-3 against the float64 oracle; cases whose outputs are unique up to
rounding order (placement, sharing, repetition) are compared bit for bit.
"""
import json
import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import paged_kv_cache_305_gb300 as pa
import workloads as W
from gpu_util import (ATOL, DeviceCase, check_parity, dev_bits, host_bits, max_err,
                      oracle_after_write)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_305_gb300 import build
    build.build()
    pa.bad_index_count(clear=True)
    yield
    torch.cuda.synchronize()


def _parity(dc, ref, pt=None, what=""):
    """Run the 16-bit and the fp32 output of the same decode and apply the parity bar."""
    out16 = host_bits(dc.decode(pt)).copy()
    out32 = dc.decode(pt, out_f32=True).cpu().numpy()
    check_parity(out16, out32, ref, dc.case.dtype, what or dc.case.name)
    return out16


def _check_step(case):
    dc = DeviceCase(case)
    dc.write_new_tokens()
    kc, vc = oracle_after_write(case)
    ref = oracle.paged_decode(case.query, kc, vc, case.block_tables, case.seq_lens,
                              case.block_size, case.scale, case.dtype)
    _parity(dc, ref)
    return dc, ref


def test_tiny_workload():
    _check_step(W.make_workload("tiny"))


GRID = [
    # dtype, d, Hq, Hkv, B, lengths, partition_tokens
    ("fp16", 64, 4, 4, 16, (1, 128), 0),
    ("bf16", 128, 32, 8, 16, (1, 700), 64),
    ("fp16", 128, 16, 1, 8, (1, 300), 0),
    ("bf16", 64, 6, 3, 4, (1, 90), 32),
    ("fp16", 128, 8, 8, 1, (1, 200), 0),
    ("bf16", 128, 16, 2, 32, (1, 1100), 0),
    ("fp16", 64, 8, 2, 64, (1, 1500), 128),
    ("bf16", 128, 12, 4, 2, (1, 100), 16),
    ("fp16", 128, 64, 8, 16, (600, 2100), 512),
    ("bf16", 64, 2, 1, 16, (1, 40), 0),
]


@pytest.mark.parametrize("idx", range(len(GRID)))
def test_random_grid(idx):
    dtype, d, Hq, Hkv, B, lens, pt = GRID[idx]
    case = W.random_case(num_seqs=5, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=lens, dtype=dtype, seed=100 + idx,
                         partition_tokens=pt, name=f"grid-{dtype}-{d}-{Hq}/{Hkv}-B{B}")
    _check_step(case)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_boundary_lengths(dtype):
    lens = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 511, 512, 513, 1023, 1024, 1025]
    case = W.random_case(num_seqs=len(lens), num_q_heads=8, num_kv_heads=2, head_dim=128,
                         block_size=16, len_range=(1, 1025), dtype=dtype, seed=3, seq_lens=lens)
    _check_step(case)


def test_worked_example_in_head_dim_64():
    # "PagedAttention by hand": d=2, B=2, table [2, 0, 1], 5 tokens, q=(1,2),
    # no scale; embedded in head_dim 64 by zero padding (dims >= 2 are zero)
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
    d = 64
    kc = np.zeros((9, 2, 1, d), np.float32)
    vc = np.zeros((9, 2, 1, d), np.float32)
    for k, rows in g["key_blocks"].items():
        kc[int(k), :, 0, :2] = rows
    for k, rows in g["value_blocks"].items():
        vc[int(k), :, 0, :2] = rows
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, :2] = g["query"]
    dt = "fp16"
    out = torch.empty((1, 1, d), dtype=torch.float16, device="cuda")
    pa.decode(out, dev_bits(W.f32_to_bits(q, dt), dt), dev_bits(W.f32_to_bits(kc, dt), dt),
              dev_bits(W.f32_to_bits(vc, dt), dt),
              torch.tensor([g["block_table"]], dtype=torch.int32, device="cuda"),
              torch.tensor([g["seq_len"]], dtype=torch.int32, device="cuda"), scale=1.0)
    got = oracle.to_float64(host_bits(out), dt)[0, 0]
    assert abs(got[0] - 4.125619931152994) <= ATOL and abs(got[1] - 4.125619931152994) <= ATOL
    assert np.all(got[2:] == 0)
    out32 = torch.empty((1, 1, d), dtype=torch.float32, device="cuda")
    pa.decode(out32, dev_bits(W.f32_to_bits(q, dt), dt), dev_bits(W.f32_to_bits(kc, dt), dt),
              dev_bits(W.f32_to_bits(vc, dt), dt),
              torch.tensor([g["block_table"]], dtype=torch.int32, device="cuda"),
              torch.tensor([g["seq_len"]], dtype=torch.int32, device="cuda"), scale=1.0)
    ref = np.zeros((1, 1, d))
    ref[0, 0, :2] = 4.125619931152994
    check_parity(host_bits(out), out32.cpu().numpy(), ref, dt, "worked example")
    # the page's printed code output, 4.1256 to 4 decimals
    assert abs(got[0] - g["printed"]["output_code_4dp"][0]) <= ATOL


@pytest.mark.parametrize("dtype,G", [("fp16", 1), ("bf16", 4), ("bf16", 8)])
def test_seq_len_one_returns_v_row_exactly(dtype, G):
    case = W.random_case(num_seqs=6, num_q_heads=2 * G, num_kv_heads=2, head_dim=128,
                         block_size=16, len_range=(1, 1), dtype=dtype, seed=G)
    dc = DeviceCase(case)
    got = host_bits(dc.decode())
    for s in range(case.num_seqs):
        v = case.value_cache[case.block_tables[s, 0], 0]
        for hq in range(case.num_q_heads):
            assert np.array_equal(got[s, hq], v[hq // G])


def test_zero_length_writes_zeros():
    case = W.random_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                         len_range=(1, 900), dtype="bf16", seed=2, seq_lens=[0, 700, 0, 33])
    dc = DeviceCase(case)
    dc.out.fill_(1.0)
    got = host_bits(dc.decode(partition_tokens=64))
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = oracle.paged_decode(case.query, case.key_cache, case.value_cache, case.block_tables,
                              case.seq_lens, 16, case.scale, "bf16")
    _parity(dc, ref, 64)


def test_unused_slots_and_table_tail_are_never_read():
    case = W.random_case(num_seqs=6, num_q_heads=8, num_kv_heads=4, head_dim=128, block_size=16,
                         len_range=(1, 600), dtype="fp16", seed=4)
    base = host_bits(DeviceCase(case).decode())
    W.poison_unused(case, W.nan_bits("fp16"))
    poisoned = host_bits(DeviceCase(case).decode())
    assert np.array_equal(base, poisoned)
    W.poison_unused(case, W.inf_bits("fp16"))
    assert np.array_equal(base, host_bits(DeviceCase(case).decode()))


def test_placement_independence_bit_exact():
    case = W.random_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=8,
                         len_range=(100, 900), dtype="bf16", seed=5)
    base = host_bits(DeviceCase(case).decode())
    perm = np.random.default_rng(1).permutation(case.num_blocks)
    kc = np.empty_like(case.key_cache)
    vc = np.empty_like(case.value_cache)
    kc[perm] = case.key_cache
    vc[perm] = case.value_cache
    case.key_cache, case.value_cache = kc, vc
    case.block_tables = perm[case.block_tables].astype(np.int32)
    assert np.array_equal(base, host_bits(DeviceCase(case).decode()))


def test_shared_blocks_bit_exact_vs_private():
    case = W.shared_prefix_case(block_size=16, groups=3, per_group=4, prefix=256,
                                suffix_range=(0, 300), num_heads=4, head_dim=128, seed=2)
    ref = oracle.paged_decode(case.query, case.key_cache, case.value_cache, case.block_tables,
                              case.seq_lens, 16, case.scale, "fp16")
    shared = _parity(DeviceCase(case), ref)
    B = 16
    ks, vs, tables = [], [], np.zeros_like(case.block_tables)
    for s in range(case.num_seqs):
        for j in range((int(case.seq_lens[s]) + B - 1) // B):
            ks.append(case.key_cache[case.block_tables[s, j]])
            vs.append(case.value_cache[case.block_tables[s, j]])
            tables[s, j] = len(ks) - 1
    case.key_cache, case.value_cache = np.stack(ks), np.stack(vs)
    case.num_blocks = len(ks)
    case.block_tables = tables
    assert np.array_equal(shared, host_bits(DeviceCase(case).decode()))


def test_repeatable_and_workspace_reusable():
    case = W.random_case(num_seqs=7, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                         len_range=(1, 3000), dtype="bf16", seed=6, partition_tokens=128)
    dc = DeviceCase(case)
    a = host_bits(dc.decode()).copy()
    b = host_bits(dc.decode()).copy()
    assert np.array_equal(a, b)
    # the header (claim counter, finished CTAs) and the arrival counters are
    # back at zero after every call
    ws = dc.workspace
    assert int(ws[: 256 + case.num_seqs * case.num_kv_heads * 4].view(torch.int32).abs().sum()) == 0
    ref = oracle.paged_decode(case.query, case.key_cache, case.value_cache, case.block_tables,
                              case.seq_lens, 16, case.scale, "bf16")
    assert np.array_equal(_parity(dc, ref), a)


def test_one_workspace_for_a_small_then_a_larger_batch():
    # A serving loop whose batch grows keeps its workspace: the larger call's
    # arrival counters then sit on bytes where the smaller call left fp32
    # partial results (its log-sum-exp values start right after its 64
    # counters). Every row of both calls is cut into pieces (many 16- or
    # 64-token partitions per row), so every row goes through a counter.
    small = W.random_case(num_seqs=2, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          len_range=(2500, 3000), dtype="bf16", seed=31, partition_tokens=16)
    big = W.random_case(num_seqs=40, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                        len_range=(2500, 3000), dtype="bf16", seed=32, partition_tokens=64)
    cases = [DeviceCase(c) for c in (small, big)]
    need = max(pa.decode_workspace_bytes(c.num_seqs, c.num_q_heads, c.head_dim,
                                         c.max_blocks_per_seq, c.block_size, c.partition_tokens)
               for c in (small, big))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    refs = [oracle.paged_decode(c.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                                c.block_size, c.scale, c.dtype) for c in (small, big)]
    for k in (0, 1, 0, 1):
        dc, c = cases[k], cases[k].case
        got = []
        for out in (dc.out, dc.out32):
            out.fill_(float("nan"))  # a row the merge never writes stays NaN
            pa.decode(out, dc.query, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens,
                      c.scale, c.partition_tokens, ws)
            got.append(out.clone())
        check_parity(host_bits(got[0]), got[1].cpu().numpy(), refs[k], c.dtype,
                     f"shared workspace, call with {c.num_seqs} sequences")
        assert np.array_equal(got[1].cpu().numpy(), dc.decode(out_f32=True).cpu().numpy())


def test_partition_length_does_not_change_the_result():
    case = W.random_case(num_seqs=4, num_q_heads=8, num_kv_heads=1, head_dim=128, block_size=16,
                         len_range=(2000, 5000), dtype="bf16", seed=7)
    ref = oracle.paged_decode(case.query, case.key_cache, case.value_cache, case.block_tables,
                              case.seq_lens, 16, case.scale, "bf16")
    dc = DeviceCase(case)
    outs = []
    for pt in (16, 64, 512, 4096, 16384):
        _parity(dc, ref, pt, f"partition_tokens={pt}")
        outs.append(dc.out32.cpu().numpy().astype(np.float64))
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= ATOL


def test_runs_on_a_side_stream():
    case = W.random_case(num_seqs=3, num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                         len_range=(1, 400), dtype="fp16", seed=8)
    dc = DeviceCase(case)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        dc.step()
    st.synchronize()
    kc, vc = oracle_after_write(case)
    ref = oracle.paged_decode(case.query, kc, vc, case.block_tables, case.seq_lens, 16,
                              case.scale, "fp16")
    out16 = host_bits(dc.out).copy()
    with torch.cuda.stream(st):
        dc.decode(out_f32=True)
    st.synchronize()
    check_parity(out16, dc.out32.cpu().numpy(), ref, "fp16", "side stream")


def test_bad_indices_are_counted_not_faulted():
    case = W.random_case(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                         len_range=(40, 100), dtype="fp16", seed=9)
    pa.bad_index_count(clear=True)
    good = host_bits(DeviceCase(case).decode()).copy()
    assert pa.bad_index_count() == 0
    case.block_tables[1, 0] = case.num_blocks + 5      # a block id outside the pool
    case.block_tables[2, 1] = -3
    case.seq_lens[0] = case.max_blocks_per_seq * 16 + 7  # longer than the table allows
    dc = DeviceCase(case)
    got = host_bits(dc.decode())
    assert pa.bad_index_count(clear=True) >= 3
    assert np.all(np.isfinite(oracle.to_float64(got, "fp16")))
    assert pa.bad_index_count() == 0


def test_small_workspace_is_rejected():
    case = W.random_case(num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                         len_range=(1, 2000), dtype="fp16", seed=10)
    dc = DeviceCase(case)
    with pytest.raises(pa.PagedAttnError, match="workspace"):
        pa.decode(dc.out, dc.query, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens,
                  case.scale, 0, dc.workspace[:64])


APPEND_CASES = [
    # dtype, d, Hq, Hkv, B, lengths, partition_tokens
    ("bf16", 128, 32, 8, 16, (1, 3000), 256),
    ("fp16", 64, 4, 4, 1, (1, 300), 0),
    ("bf16", 128, 16, 1, 64, (1, 900), 128),
    ("fp16", 128, 8, 2, 8, (1, 40), 16),
]


@pytest.mark.parametrize("idx", range(len(APPEND_CASES)))
def test_decode_append_equals_write_then_decode(idx):
    dtype, d, Hq, Hkv, B, lens, pt = APPEND_CASES[idx]
    case = W.random_case(num_seqs=9, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=lens, dtype=dtype, seed=300 + idx, partition_tokens=pt)
    case.seq_lens[3] = 0  # nothing to write, zero output
    case.slot_mapping[3] = -1
    two = DeviceCase(case)
    two.write_new_tokens()
    want16 = host_bits(two.decode()).copy()
    want32 = two.decode(out_f32=True).cpu().numpy().copy()
    one = DeviceCase(case)
    for out, want in ((one.out, None), (one.out32, want32)):
        pa.decode_append(out, one.query, one.new_key, one.new_value, one.key_cache, one.value_cache,
                         one.block_tables, one.seq_lens, case.scale, pt, one.workspace)
    assert np.array_equal(host_bits(one.out), want16)
    assert np.array_equal(one.out32.cpu().numpy(), want32)
    assert np.array_equal(host_bits(one.key_cache), host_bits(two.key_cache))
    assert np.array_equal(host_bits(one.value_cache), host_bits(two.value_cache))
    kc, vc = oracle_after_write(case)
    ref = oracle.paged_decode(case.query, kc, vc, case.block_tables, case.seq_lens, B,
                              case.scale, dtype)
    check_parity(want16, want32, ref, dtype, "decode_append")
