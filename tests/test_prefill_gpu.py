"""GPU parity of pa_prefill (paged causal prefill, through the C ABI) against
the float64 oracle: chunks of new tokens of several lengths (one token, part
of a prompt, a whole prompt), several query tiles and key tiles per sequence,
ragged tails, every group size path and block size."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import paged_kv_cache_305_gb300 as pa
import workloads as W
from gpu_util import ATOL, DeviceCase, check_parity, dev_bits, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_305_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def _ws(dc, use=True):
    """The prefill workspace (bf16: fp16 copy of the value rows), or None."""
    return pa.alloc_prefill_workspace(dc.seq_lens, dc.key_cache, dc.block_tables) if use else None


def _run(case, qlens, seed, scale=None, workspace=True):
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = W.normal_bits((int(starts[-1]), case.num_q_heads, case.head_dim), case.dtype, seed, 55)
    dc = DeviceCase(case)
    qd = dev_bits(q, case.dtype)
    qs = torch.from_numpy(starts).cuda()
    out16 = torch.empty_like(qd)
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    mq = int(max(qlens))
    sc = case.scale if scale is None else scale
    ws = _ws(dc, workspace)
    pa.prefill(out16, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs, mq, sc, ws)
    pa.prefill(out32, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs, mq, sc, ws)
    ref = oracle.paged_prefill(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                               starts, case.block_size, sc, case.dtype)
    assert pa.wait_timeout_count(clear=True) == 0
    check_parity(host_bits(out16), out32.cpu().numpy(), ref, case.dtype, f"prefill {case.name}")
    return q, out32.cpu().numpy()


CASES = [
    # dtype, d, Hq, Hkv, B, lengths
    ("bf16", 128, 32, 8, 16, (40, 700)),
    ("fp16", 64, 4, 4, 1, (1, 200)),
    ("bf16", 128, 16, 1, 64, (100, 500)),
    ("fp16", 128, 12, 4, 8, (1, 150)),
    ("bf16", 64, 16, 2, 16, (70, 300)),
    ("fp16", 128, 16, 1, 4, (50, 300)),   # row copies (B < 8), 16 query heads per kv head
    ("bf16", 128, 24, 8, 32, (90, 400)),  # tensor-core kernel, 3 heads per kv head, B = 32
    ("bf16", 64, 8, 8, 64, (60, 600)),    # d = 64 (one head-dim slice per box), whole 64-token blocks
    ("fp16", 64, 32, 4, 8, (30, 400)),    # d = 64, 8-token blocks, 8 query heads per kv head
]


@pytest.mark.parametrize("idx", range(len(CASES)))
@pytest.mark.parametrize("workspace", [True, False])
def test_prefill_chunks(idx, workspace):
    # bf16 with a workspace: the value rows converted to fp16, one P.V
    # product; without: the two-product path (fp16 needs no workspace)
    dtype, d, Hq, Hkv, B, lens = CASES[idx]
    if dtype == "fp16" and not workspace:
        pytest.skip("fp16 takes no workspace")
    case = W.random_case(num_seqs=5, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=lens, dtype=dtype, seed=400 + idx)
    L = case.seq_lens
    # a whole prompt, one token, a partial chunk, a zero-length chunk, a ragged chunk
    qlens = [int(L[0]), 1, max(1, int(L[2]) // 3), 0, min(int(L[4]), 77)]
    _run(case, qlens, idx, workspace=workspace)


def test_single_token_chunks_match_decode():
    case = W.random_case(num_seqs=6, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                         len_range=(1, 900), dtype="bf16", seed=7)
    q, got = _run(case, [1] * 6, 3)
    dc = DeviceCase(case)
    out32 = torch.empty((6, 32, 128), dtype=torch.float32, device="cuda")
    pa.decode(out32, dev_bits(q, "bf16"), dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens,
              case.scale, 0, dc.workspace)
    assert np.max(np.abs(out32.cpu().numpy() - got)) <= ATOL


def test_long_prompt_many_tiles():
    case = W.random_case(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                         len_range=(1500, 1500), dtype="bf16", seed=8)
    _run(case, [1500, 1000], 5)


@pytest.mark.parametrize("B", [16, 4])
def test_many_sequences_ragged_chunks(B):
    # thousands of (query tile, kv head, sequence) CTAs, several waves per SM,
    # chunks of every length (some empty, some whole prompts); B = 4 takes
    # the row-copy producers
    case = W.random_case(num_seqs=48, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=B,
                         len_range=(1, 400), dtype="bf16", seed=90 + B)
    qlens = [int(x) if i % 3 else int(x) // 2 for i, x in enumerate(case.seq_lens)]
    qlens[5] = 0
    _run(case, qlens, 13)


@pytest.mark.parametrize("B", [8, 16, 64, 2])
def test_unused_slots_are_never_read(B):
    # tail slots of each last block and blocks outside the tables hold NaN / Inf:
    # the output must not change (rows past L are zero-filled, never loaded)
    case = W.random_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=B,
                         len_range=(3, 260), dtype="bf16", seed=30 + B)
    qlens = [int(x) for x in np.minimum(case.seq_lens, 97)]
    _, base = _run(case, qlens, 11)
    W.poison_unused(case, W.nan_bits("bf16"))
    _, nan_out = _run(case, qlens, 11)
    W.poison_unused(case, W.inf_bits("bf16"))
    _, inf_out = _run(case, qlens, 11)
    assert np.array_equal(base, nan_out) and np.array_equal(base, inf_out)


@pytest.mark.parametrize("B", [16, 2])
def test_bad_block_ids_are_counted_not_faulted(B):
    case = W.random_case(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=B,
                         len_range=(100, 200), dtype="bf16", seed=41)
    starts = np.array([0, 10, 20, 30], dtype=np.int32)
    dc = DeviceCase(case)
    bt = dc.block_tables.clone()
    bt[1, 2] = case.num_blocks + 5   # inside sequence 1's length: read as zeros
    bt[2, 0] = -3
    q = dev_bits(W.normal_bits((30, 8, 128), "bf16", 5, 55), "bf16")
    out = torch.empty((30, 8, 128), dtype=torch.float32, device="cuda")
    pa.bad_index_count(clear=True)
    pa.prefill(out, q, dc.key_cache, dc.value_cache, bt, dc.seq_lens, torch.from_numpy(starts).cuda(),
               10, case.scale, _ws(dc))
    assert pa.bad_index_count(clear=True) >= 2
    assert pa.wait_timeout_count(clear=True) == 0
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("B", [16, 4])
@pytest.mark.parametrize("scale", [-0.3, 0.0, 1.5])
def test_scale_sign_and_zero(B, scale):
    # a negative scale flips which token dominates; zero gives the plain mean
    # of the visible values
    case = W.random_case(num_seqs=3, num_q_heads=8, num_kv_heads=4, head_dim=64, block_size=B,
                         len_range=(20, 180), dtype="fp16", seed=50 + B)
    _run(case, [int(x) for x in case.seq_lens], 12, scale=scale)


@pytest.mark.parametrize("B", [64, 16])
def test_repeated_calls_are_bit_identical(B):
    # the tensor-core kernel's warps hand tiles to each other through shared-
    # memory barriers; a missing or early signal shows up as run-to-run
    # differences, so the same call is repeated and compared bit for bit
    case = W.random_case(num_seqs=5, num_q_heads=16, num_kv_heads=1, head_dim=128, block_size=B,
                         len_range=(100, 500), dtype="bf16", seed=402)
    L = case.seq_lens
    qlens = [int(L[0]), 1, max(1, int(L[2]) // 3), 0, min(int(L[4]), 77)]
    q0, first = _run(case, qlens, 2)
    starts = torch.from_numpy(np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)).cuda()
    dc = DeviceCase(case)
    qd = dev_bits(q0, "bf16")
    ws = _ws(dc)
    for _ in range(24):
        out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
        pa.prefill(out, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, starts,
                   max(qlens), case.scale, ws)
        assert np.array_equal(out.cpu().numpy(), first)
    assert pa.wait_timeout_count(clear=True) == 0


@pytest.mark.parametrize("ctx", [4096, 2048])
def test_full_size_chunked_prefill_sampled(ctx):
    # the configurations bench.py times: 16 sequences, 32/8 heads, d = 128,
    # block size 16, bf16, a 2048-token chunk after 2048 cached tokens, and
    # whole 2048-token prompts; the oracle computes sampled (sequence,
    # position, kv head) outputs one by one. At this size both CTAs of every
    # SM and all the product / softmax hand-overs run under full contention,
    # so the call is also repeated: every repeat must be bit-identical and no
    # bounded wait may give up.
    S, Hq, Hkv, d, B, chunk = 16, 32, 8, 128, 16, 2048
    case = W.random_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=(ctx, ctx), dtype="bf16", seed=0)
    starts = np.arange(0, (S + 1) * chunk, chunk, dtype=np.int32)
    q = W.normal_bits((S * chunk, Hq, d), "bf16", 1, 55)
    dc = DeviceCase(case)
    qd = dev_bits(q, "bf16")
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    out16 = torch.empty_like(qd)
    qs = torch.from_numpy(starts).cuda()
    ws = _ws(dc)
    pa.prefill(out32, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs, chunk, case.scale, ws)
    pa.prefill(out16, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs, chunk, case.scale, ws)
    assert pa.wait_timeout_count(clear=True) == 0
    got32 = out32.cpu().numpy()
    got16 = host_bits(out16)
    again = torch.empty_like(out32)
    for _ in range(8):
        again.fill_(float("nan"))
        pa.prefill(again, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs, chunk,
                   case.scale, ws)
        assert torch.equal(again, out32)
    assert pa.wait_timeout_count(clear=True) == 0
    del again
    del dc, qd, out32, out16, ws
    torch.cuda.empty_cache()
    assert np.all(np.isfinite(got32))
    assert np.array_equal(oracle.round_to_dtype(got32.astype(np.float64), "bf16"), got16)
    rng = np.random.default_rng(3)
    G = Hq // Hkv
    picks = {(0, 0, 0), (S - 1, chunk - 1, Hkv - 1), (5, 63, 2), (5, 64, 2), (7, 127, 3), (7, 128, 3)}
    while len(picks) < 40:
        picks.add((int(rng.integers(S)), int(rng.integers(chunk)), int(rng.integers(Hkv))))
    err = 0.0
    for s in sorted({p[0] for p in picks}):
        L = int(case.seq_lens[s])
        K = oracle.to_float64(oracle.gather_kv(case.key_cache, case.block_tables[s], L, B), "bf16")
        V = oracle.to_float64(oracle.gather_kv(case.value_cache, case.block_tables[s], L, B), "bf16")
        for (_, j, h) in [p for p in sorted(picks) if p[0] == s]:
            pos = L - chunk + j
            qrow = oracle.to_float64(q[starts[s] + j, h * G:(h + 1) * G], "bf16")
            ref, _ = oracle.single_query_attention(qrow, K[:pos + 1, h], V[:pos + 1, h], case.scale)
            err = max(err, float(np.max(np.abs(got32[starts[s] + j, h * G:(h + 1) * G] - ref))))
    assert err <= ATOL, f"full-size prefill: max |fp32 - oracle| over sampled rows = {err}"


@pytest.mark.parametrize("B", [16, 4])
def test_a_wait_that_runs_out_is_counted_and_the_device_stays_usable(B):
    # The test hook makes each CTA's product thread wait on a barrier that
    # nothing signals: that bounded wait gives up (about one second), the
    # warps waiting for products give up after it, and every CTA winds down.
    # The call must return, the give-ups must be counted, and the next normal
    # call on the same device must give the bits of a fresh run.
    case = W.random_case(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=B,
                         len_range=(150, 300), dtype="bf16", seed=60 + B)
    qlens = [int(case.seq_lens[0]), 70]
    q0, fresh = _run(case, qlens, 13)
    starts = torch.from_numpy(np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)).cuda()
    dc = DeviceCase(case)
    qd = dev_bits(q0, "bf16")
    pa.wait_timeout_count(clear=True)
    stalled = torch.full(qd.shape, 7.0, dtype=torch.float32, device="cuda")
    ws = _ws(dc)
    pa.testing_prefill_stalled(stalled, qd, dc.key_cache, dc.value_cache, dc.block_tables,
                               dc.seq_lens, starts, max(qlens), case.scale, ws)
    assert pa.wait_timeout_count(clear=True) >= 1
    assert bool((stalled == 7.0).all())  # no product ran, nothing was stored
    out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    pa.prefill(out, qd, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, starts,
               max(qlens), case.scale, ws)
    assert np.array_equal(out.cpu().numpy(), fresh)
    assert pa.wait_timeout_count(clear=True) == 0
