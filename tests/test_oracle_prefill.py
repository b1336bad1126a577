"""Pins for the oracle's paged causal prefill.

* one new token per sequence is exactly the decode oracle;
* scalar-loop brute force with direct table addressing and an explicit causal
  limit on tiny inputs;
* causality: K/V at positions after a query never change its output;
* a full-prompt chunk equals running decode at every prefix length.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W


def _case(seed, S=3, Hq=4, Hkv=2, d=8, B=4, lens=(3, 30), dtype="bf16"):
    return W.random_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=lens, dtype=dtype, seed=seed)


def _queries(case, qlens, seed):
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = W.normal_bits((int(starts[-1]), case.num_q_heads, case.head_dim), case.dtype, seed, 77)
    return q, starts


def test_single_new_token_is_decode():
    case = _case(1)
    q, starts = _queries(case, [1] * case.num_seqs, 1)
    got = oracle.paged_prefill(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                               starts, case.block_size, case.scale, case.dtype)
    want = oracle.paged_decode(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                               case.block_size, case.scale, case.dtype)
    assert np.array_equal(got, want)


def _brute(q, kc, vc, table, lens, starts, B, scale, dtype):
    qf, kf, vf = (oracle.to_float64(x, dtype) for x in (q, kc, vc))
    Hq, d = q.shape[1], q.shape[2]
    Hkv = kc.shape[2]
    G = Hq // Hkv
    out = np.zeros(q.shape)
    for s in range(len(lens)):
        L, q0, q1 = int(lens[s]), int(starts[s]), int(starts[s + 1])
        for j in range(q1 - q0):
            limit = L - (q1 - q0) + j  # last visible position
            for hq in range(Hq):
                h = hq // G
                sc = []
                for t in range(limit + 1):
                    blk, off = int(table[s][t // B]), t % B
                    sc.append(scale * sum(float(qf[q0 + j, hq, i]) * float(kf[blk, off, h, i]) for i in range(d)))
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                for i in range(d):
                    out[q0 + j, hq, i] = math.fsum(w[t] * float(vf[int(table[s][t // B]), t % B, h, i])
                                                   for t in range(limit + 1)) / math.fsum(w)
    return out


@pytest.mark.parametrize("B,qlens", [(1, [1, 3, 2]), (4, [3, 5, 1]), (2, [2, 2, 2])])
def test_brute_force_causal(B, qlens):
    case = _case(10 + B, B=B, lens=(6, 20))
    q, starts = _queries(case, qlens, B)
    args = (q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens, starts,
            B, case.scale, case.dtype)
    assert np.allclose(oracle.paged_prefill(*args), _brute(*args), rtol=1e-12, atol=1e-13)


def test_later_tokens_do_not_change_earlier_queries():
    case = _case(20, lens=(20, 30))
    qlens = [5, 7, 3]
    q, starts = _queries(case, qlens, 3)
    base = oracle.paged_prefill(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                                starts, case.block_size, case.scale, case.dtype)
    s, B = 1, case.block_size
    L, Q = int(case.seq_lens[s]), qlens[s]
    j = 2
    p = L - Q + j
    for t in range(p + 1, L):  # perturb every token after query j's position
        case.key_cache[case.block_tables[s, t // B], t % B] ^= 0x1234
        case.value_cache[case.block_tables[s, t // B], t % B] ^= 0x0F0F
    got = oracle.paged_prefill(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                               starts, case.block_size, case.scale, case.dtype)
    row = int(starts[s]) + j
    assert np.array_equal(got[row], base[row])
    assert not np.array_equal(got[row + 1], base[row + 1])


def test_whole_prompt_chunk_equals_decode_at_every_length():
    case = _case(30, S=1, lens=(9, 9))
    L = int(case.seq_lens[0])
    q, starts = _queries(case, [L], 4)
    got = oracle.paged_prefill(q, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
                               starts, case.block_size, case.scale, case.dtype)
    for j in range(L):
        want = oracle.paged_decode(q[j:j + 1], case.key_cache, case.value_cache, case.block_tables,
                                   np.array([j + 1], np.int32), case.block_size, case.scale, case.dtype)
        assert np.array_equal(got[j], want[0])
