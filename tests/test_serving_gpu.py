"""The serving-side pieces around decode, on the GPU and through the C ABI:
pa_copy_blocks (bit-exact against the oracle's block copy) and a simulated
serving loop -- prompts, forked candidates that share their prompt blocks,
divergent decode steps with copy-on-write, freed sequences whose blocks are
reused -- where every decode is checked against attention over each
sequence's own logical token history ("PagedAttention by hand", Why divide
memory into physical blocks?: sharing with copy-on-write leaves every
candidate's attention unchanged)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import paged_kv_cache_305_gb300 as pa
import workloads as W
from gpu_util import ATOL, check_parity, dev_bits, host_bits
from oracle.block_manager import copy_blocks as oracle_copy_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_305_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype,B,Hkv,d", [("bf16", 16, 8, 128), ("fp16", 1, 4, 64), ("bf16", 64, 2, 128)])
def test_copy_blocks_bit_exact(dtype, B, Hkv, d):
    NB = 40
    kc = W.normal_bits((NB, B, Hkv, d), dtype, 7, 1)
    vc = W.normal_bits((NB, B, Hkv, d), dtype, 7, 2)
    pairs = [(3, 10), (11, 0), (39, 5), (7, 7)]
    kd, vd = dev_bits(kc, dtype), dev_bits(vc, dtype)
    src = torch.tensor([p[0] for p in pairs], dtype=torch.int32, device="cuda")
    dst = torch.tensor([p[1] for p in pairs], dtype=torch.int32, device="cuda")
    pa.copy_blocks(kd, vd, src, dst)
    oracle_copy_blocks(kc, vc, pairs)
    assert np.array_equal(host_bits(kd), kc) and np.array_equal(host_bits(vd), vc)


def test_copy_blocks_skips_out_of_range_ids():
    kd = dev_bits(W.normal_bits((4, 16, 2, 64), "fp16", 1, 1), "fp16")
    vd = dev_bits(W.normal_bits((4, 16, 2, 64), "fp16", 1, 2), "fp16")
    before = host_bits(kd).copy()
    pa.bad_index_count(clear=True)
    pa.copy_blocks(kd, vd, torch.tensor([9, -1], dtype=torch.int32, device="cuda"),
                   torch.tensor([0, 1], dtype=torch.int32, device="cuda"))
    assert pa.bad_index_count(clear=True) == 2
    assert np.array_equal(host_bits(kd), before)


@pytest.mark.parametrize("dtype,B,Hq,Hkv,d", [("bf16", 16, 32, 8, 128), ("fp16", 2, 4, 4, 64),
                                               ("bf16", 1, 8, 2, 128)])
def test_serving_loop_with_forks_and_copy_on_write(dtype, B, Hq, Hkv, d):
    rng = np.random.default_rng(B * 100 + Hq)
    NB, MB = 400, 64 // B * 8
    bm = pa.BlockManager(NB, B, MB)
    kc = torch.zeros((NB, B, Hkv, d), dtype=torch.float16 if dtype == "fp16" else torch.bfloat16,
                     device="cuda")
    vc = torch.zeros_like(kc)
    hist = {}  # sequence -> list of (k, v) rows [Hkv, d] bit patterns, logical order
    counter = [0]

    def rows(n):
        counter[0] += 1
        return (W.normal_bits((n, Hkv, d), dtype, 99, 2 * counter[0]),
                W.normal_bits((n, Hkv, d), dtype, 99, 2 * counter[0] + 1))

    def write(requests, ks, vs):
        slots, copies = bm.append(requests)
        if copies:
            pa.copy_blocks(kc, vc, torch.tensor([c[0] for c in copies], dtype=torch.int32, device="cuda"),
                           torch.tensor([c[1] for c in copies], dtype=torch.int32, device="cuda"))
        pa.reshape_and_cache(dev_bits(ks, dtype), dev_bits(vs, dtype), kc, vc,
                             torch.from_numpy(slots).cuda())
        return copies

    def check(live):
        tables, lens = bm.block_tables(live)
        q = W.normal_bits((len(live), Hq, d), dtype, 98, counter[0])
        counter[0] += 1
        out16 = torch.empty((len(live), Hq, d), dtype=kc.dtype, device="cuda")
        out32 = torch.empty((len(live), Hq, d), dtype=torch.float32, device="cuda")
        bt = torch.from_numpy(tables).cuda()
        sl = torch.from_numpy(lens).cuda()
        ws = pa.alloc_workspace(out16, kc, bt, 32)
        scale = 1 / np.sqrt(d)
        pa.decode(out16, dev_bits(q, dtype), kc, vc, bt, sl, scale, 32, ws)
        pa.decode(out32, dev_bits(q, dtype), kc, vc, bt, sl, scale, 32, ws)
        G = Hq // Hkv
        ref = np.zeros((len(live), Hq, d))
        for i, s in enumerate(live):
            K = oracle.to_float64(np.stack([r[0] for r in hist[s]]), dtype)
            V = oracle.to_float64(np.stack([r[1] for r in hist[s]]), dtype)
            qf = oracle.to_float64(q[i], dtype)
            for h in range(Hkv):
                o, _ = oracle.single_query_attention(qf[h * G:(h + 1) * G], K[:, h], V[:, h], scale)
                ref[i, h * G:(h + 1) * G] = o
        check_parity(host_bits(out16), out32.cpu().numpy(), ref, dtype, "serving loop")

    # prompts
    live = []
    for _ in range(4):
        s = bm.new_sequence()
        n = int(rng.integers(1, 40))
        ks, vs = rows(n)
        write([(s, n)], ks, vs)
        hist[s] = list(zip(ks, vs))
        live.append(s)
    # candidates sharing each prompt
    for p in list(live):
        for _ in range(int(rng.integers(1, 3))):
            c = bm.fork(p)
            hist[c] = list(hist[p])
            live.append(c)
    check(live)
    total_copies = 0
    for step in range(12):
        ks, vs = rows(len(live))
        total_copies += len(write([(s, 1) for s in live], ks, vs))
        for i, s in enumerate(live):
            hist[s].append((ks[i], vs[i]))
        if step % 4 == 3:
            check(live)
        if step == 5:  # finish two candidates, start a new prompt in their blocks
            for s in (live.pop(1), live.pop(2)):
                bm.free_sequence(s)
                del hist[s]
            s = bm.new_sequence()
            ks, vs = rows(25)
            write([(s, 25)], ks, vs)
            hist[s] = list(zip(ks, vs))
            live.append(s)
    check(live)
    if B > 1:
        assert total_copies > 0  # the forks really diverged through copy-on-write
    else:
        assert total_copies == 0  # one-token blocks are never written once shared
