"""The library's calls inside CUDA graphs: a captured decode step (fused cache
write + attention) and a captured prefill, replayed several times, give the
same bits as the same calls made directly. Every call takes the caller's
current stream and makes no host synchronisation, and the split-K arrival
counters are left at zero by each launch, so a replayed graph needs nothing
re-initialised."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

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


@pytest.mark.parametrize("name", ["tiny", "llama2_7b_mha"])
def test_captured_decode_step_replays_bit_identically(name):
    case = W.make_workload(name)
    dc = DeviceCase(case)
    pt = dc.partition_tokens or 64  # several partitions: the split-K merge runs inside the graph
    ws = pa.alloc_workspace(dc.query, dc.key_cache, dc.block_tables, pt)
    out = torch.empty_like(dc.query)

    def step():
        pa.decode_append(out, dc.query, dc.new_key, dc.new_value, dc.key_cache, dc.value_cache,
                         dc.block_tables, dc.seq_lens, case.scale, pt, ws)

    step()  # direct call (also fills the launch-plan cache before capture)
    torch.cuda.synchronize()
    want = host_bits(out).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), want)
    assert pa.bad_index_count(clear=True) == 0


@pytest.mark.parametrize("workspace", [True, False])
def test_captured_prefill_replays_bit_identically(workspace):
    # with a workspace the call is two kernels (the fp16 copy of the value
    # rows, then the prefill); both are captured
    case = W.random_case(num_seqs=4, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                         len_range=(100, 600), dtype="bf16", seed=9)
    qlens = [int(x) for x in np.minimum(case.seq_lens, 200)]
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = dev_bits(W.normal_bits((int(starts[-1]), 16, 128), "bf16", 9, 55), "bf16")
    dc = DeviceCase(case)
    qs = torch.from_numpy(starts).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = pa.alloc_prefill_workspace(dc.seq_lens, dc.key_cache, dc.block_tables) if workspace else None

    def call():
        pa.prefill(out, q, dc.key_cache, dc.value_cache, dc.block_tables, dc.seq_lens, qs,
                   max(qlens), case.scale, ws)

    call()
    torch.cuda.synchronize()
    want = out.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want)
    assert pa.wait_timeout_count(clear=True) == 0
