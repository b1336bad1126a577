"""Pins for the CPU oracle: each check compares it with something other than itself.

* the worked example printed in "PagedAttention by hand" (tests/golden);
* closed forms written from the mathematics;
* brute force with scalar Python loops that address each token directly
  (``table[t // B]``, offset ``t % B``) instead of gathering;
* the invariants the pages state: placement does not matter, shared blocks
  give the same result as private copies, weights sum to one, masked slots
  weigh zero, a one-token sequence returns its V row.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _bits(x, dtype):
    return W.f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


def _worked_example(dtype="fp16"):
    g = json.load(open(GOLDEN))
    NB, B, d = g["num_blocks"], g["block_size"], g["head_dim"]
    kc = np.zeros((NB, B, 1, d), np.float32)
    vc = np.zeros((NB, B, 1, d), np.float32)
    for k, rows in g["key_blocks"].items():
        kc[int(k), :, 0] = rows
    for k, rows in g["value_blocks"].items():
        vc[int(k), :, 0] = rows
    q = np.array(g["query"], np.float32).reshape(1, 1, d)
    table = np.array([g["block_table"]], np.int32)
    lens = np.array([g["seq_len"]], np.int32)
    return g, _bits(q, dtype), _bits(kc, dtype), _bits(vc, dtype), table, lens


# ---------------------------------------------------------------------------
# The printed worked example
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_worked_example_output(dtype):
    g, q, kc, vc, table, lens = _worked_example(dtype)
    out = oracle.paged_decode(q, kc, vc, table, lens, g["block_size"], g["scale"], dtype)
    # the code's output is printed to 4 decimals: 4.1256 for both dims
    for v, printed in zip(out[0, 0], g["printed"]["output_code_4dp"]):
        assert abs(v - printed) <= 0.5e-4 + 1e-12
    # the hand calculation rounds every probability to 4 decimals (4.1259)
    p4 = np.array(g["printed"]["probs_4dp"])
    hand = p4 @ np.array([1, 2, 3, 4, 5], dtype=np.float64)
    assert abs(hand - g["printed"]["output_hand_4dp"][0]) <= 0.5e-4 + 1e-12
    # closed form from the page's scores [1,2,3,2,4] and V rows 1..5
    e = [math.exp(s) for s in g["printed"]["scores"]]
    exact = sum(w * v for w, v in zip(e, [1, 2, 3, 4, 5])) / sum(e)
    assert abs(out[0, 0, 0] - exact) <= 1e-12 and abs(out[0, 0, 1] - exact) <= 1e-12
    assert abs(exact - 4.125619931152994) <= 1e-12


def test_worked_example_scores_and_probs():
    g, q, kc, vc, table, lens = _worked_example()
    K = oracle.to_float64(oracle.gather_kv(kc, table[0], 5, 2), "fp16")[:, 0, :]
    V = oracle.to_float64(oracle.gather_kv(vc, table[0], 5, 2), "fp16")[:, 0, :]
    assert K.shape == (5, 2)
    o, p = oracle.single_query_attention(np.array([1.0, 2.0]), K, V, 1.0)
    assert np.all(np.abs(p - np.array(g["printed"]["probs_4dp"])) <= 0.5e-4 + 1e-12)
    # scores are recovered from log-probability differences
    scores = np.log(p) - np.log(p[4]) + 4.0
    assert np.allclose(scores, g["printed"]["scores"], atol=1e-12, rtol=0)
    # Step 3's printed sum of exponentials after subtracting the max (4)
    assert abs(np.sum(np.exp(np.array(g["printed"]["scores"]) - 4.0)) - g["printed"]["exp_sum_4dp"]) <= 0.5e-4
    assert abs(np.sum(p) - 1.0) <= 1e-15


def test_step2_masking_gives_zero_weight():
    # Step 2 masks the 6th slot with -inf; its weight must be exactly zero
    p = oracle.attention_weights(np.array([1.0, 2.0, 3.0, 2.0, 4.0, -np.inf]))
    assert p[5] == 0.0
    assert abs(p.sum() - 1.0) <= 1e-15
    # leaving it at 0 instead shifts the weights by about 1% (the page's warning)
    q = oracle.attention_weights(np.array([1.0, 2.0, 3.0, 2.0, 4.0, 0.0]))
    assert 0.005 < q[5] < 0.015


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scale", [1.0, 0.125, 1 / math.sqrt(64)])
def test_two_token_closed_form(scale):
    # q = (a, 0), K rows (1, 0) and (0, 0): scores (a*scale, 0)
    a = 3.0
    q = np.array([a, 0.0])
    K = np.array([[1.0, 0.0], [0.0, 0.0]])
    V = np.array([[2.0, -1.0], [-4.0, 0.5]])
    o, p = oracle.single_query_attention(q, K, V, scale)
    p0 = 1.0 / (1.0 + math.exp(-a * scale))
    assert abs(p[0] - p0) <= 1e-15 and abs(p[1] - (1 - p0)) <= 1e-15
    assert np.allclose(o, p0 * V[0] + (1 - p0) * V[1], atol=1e-14, rtol=0)


def test_uniform_scores_average_values():
    # equal keys give equal weights: the output is the mean of the V rows
    K = np.ones((7, 4))
    V = np.arange(28, dtype=np.float64).reshape(7, 4)
    o, p = oracle.single_query_attention(np.array([0.3, -1.0, 2.0, 0.5]), K, V, 0.7)
    assert np.allclose(p, 1 / 7, atol=1e-15)
    assert np.allclose(o, V.mean(axis=0), atol=1e-12)


# ---------------------------------------------------------------------------
# Brute force with scalar loops
# ---------------------------------------------------------------------------
def _brute_force(q, kc, vc, table, lens, B, scale, dtype):
    qf, kf, vf = (oracle.to_float64(x, dtype) for x in (q, kc, vc))
    S, Hq, d = q.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((S, Hq, d))
    for s in range(S):
        L = int(lens[s])
        for hq in range(Hq):
            h = hq // G
            sc = []
            for t in range(L):
                blk = int(table[s][t // B])
                off = t % B
                acc = 0.0
                for i in range(d):
                    acc += float(qf[s, hq, i]) * float(kf[blk, off, h, i])
                sc.append(acc * scale)
            if not sc:
                continue
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            tot = math.fsum(w)
            for i in range(d):
                num = math.fsum(w[t] * float(vf[int(table[s][t // B]), t % B, h, i]) for t in range(L))
                out[s, hq, i] = num / tot
    return out


@pytest.mark.parametrize("B,Hq,Hkv,d,dtype", [(1, 2, 2, 4, "fp16"), (2, 4, 2, 8, "bf16"),
                                               (4, 4, 1, 8, "fp16"), (4, 6, 3, 2, "bf16")])
def test_brute_force_random(B, Hq, Hkv, d, dtype):
    case = W.random_case(num_seqs=4, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                         block_size=B, len_range=(1, 20), dtype=dtype, seed=B * 7 + d)
    # include block-boundary lengths
    case.seq_lens[:] = np.minimum(case.seq_lens, case.max_blocks_per_seq * B)
    args = (case.query, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
            B, case.scale, dtype)
    got = oracle.paged_decode(*args)
    ref = _brute_force(*args)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("lens", [[1, 3, 4, 5], [8, 7, 9, 16]])
def test_brute_force_boundary_lengths(lens):
    case = W.random_case(num_seqs=4, num_q_heads=2, num_kv_heads=2, head_dim=4,
                         block_size=4, len_range=(1, 16), dtype="fp16", seed=3, seq_lens=lens)
    args = (case.query, case.key_cache, case.value_cache, case.block_tables, case.seq_lens,
            4, case.scale, "fp16")
    assert np.allclose(oracle.paged_decode(*args), _brute_force(*args), rtol=1e-12, atol=1e-13)


def test_demo_shape_scattered_blocks():
    # "Demonstration with Non-Contiguous Blocks": 8 blocks of 4, 2 heads,
    # head_dim 8, lengths 10 and 7, tables [0,3,5,0,...] and [1,7,0,...]
    rng = np.random.default_rng(42)
    kc = W.f32_to_bits(rng.standard_normal((8, 4, 2, 8), dtype=np.float32), "fp16")
    vc = W.f32_to_bits(rng.standard_normal((8, 4, 2, 8), dtype=np.float32), "fp16")
    q = W.f32_to_bits(rng.standard_normal((2, 2, 8), dtype=np.float32), "fp16")
    table = np.array([[0, 3, 5, 0, 0, 0, 0, 0], [1, 7, 0, 0, 0, 0, 0, 0]], np.int32)
    lens = np.array([10, 7], np.int32)
    args = (q, kc, vc, table, lens, 4, 1 / math.sqrt(8), "fp16")
    out = oracle.paged_decode(*args)
    assert out.shape == (2, 2, 8)
    assert np.allclose(out, _brute_force(*args), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
def _small_case(seed=5, B=4, dtype="bf16", Hq=4, Hkv=2):
    return W.random_case(num_seqs=3, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=8,
                         block_size=B, len_range=(1, 30), dtype=dtype, seed=seed)


def _run(case, kc=None, vc=None, table=None):
    return oracle.paged_decode(case.query, case.key_cache if kc is None else kc,
                               case.value_cache if vc is None else vc,
                               case.block_tables if table is None else table,
                               case.seq_lens, case.block_size, case.scale, case.dtype)


def test_placement_independence():
    case = _small_case()
    base = _run(case)
    perm = np.random.default_rng(9).permutation(case.num_blocks)
    kc = np.empty_like(case.key_cache)
    vc = np.empty_like(case.value_cache)
    kc[perm] = case.key_cache
    vc[perm] = case.value_cache
    moved = _run(case, kc, vc, perm[case.block_tables].astype(np.int32))
    assert np.array_equal(base, moved)


def test_shared_blocks_equal_private_copies():
    case = W.shared_prefix_case(block_size=4, groups=2, per_group=3, prefix=8,
                                suffix_range=(0, 6), num_heads=2, head_dim=8, seed=4)
    shared = _run(case)
    # give every sequence private copies of all its blocks
    B = case.block_size
    rows_k, rows_v, tables = [], [], np.zeros_like(case.block_tables)
    nxt = 0
    for s in range(case.num_seqs):
        nb = (int(case.seq_lens[s]) + B - 1) // B
        for j in range(nb):
            rows_k.append(case.key_cache[case.block_tables[s, j]])
            rows_v.append(case.value_cache[case.block_tables[s, j]])
            tables[s, j] = nxt
            nxt += 1
    private = _run(case, np.stack(rows_k), np.stack(rows_v), tables)
    assert np.array_equal(shared, private)
    # and the sharing is real: group members point at the same prefix blocks
    assert np.array_equal(case.block_tables[0, :2], case.block_tables[1, :2])


def test_block_size_invariance():
    outs = []
    for B in (1, 2, 4, 8, 16):
        case = W.shared_prefix_case(block_size=B, groups=2, per_group=2, prefix=16,
                                    suffix_range=(0, 9), num_heads=2, head_dim=8, seed=6)
        outs.append(_run(case))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_unused_slots_are_never_read():
    case = _small_case(seed=8)
    base = _run(case)
    W.poison_unused(case, W.nan_bits(case.dtype))
    # also poison the junk tail of every table with another (valid) id
    assert np.array_equal(base, _run(case))
    assert np.all(np.isfinite(base))


def test_seq_len_one_returns_v_exactly():
    case = _small_case(seed=10, dtype="fp16")
    case.seq_lens[:] = 1
    out = _run(case)
    G = case.group
    for s in range(case.num_seqs):
        v = oracle.to_float64(case.value_cache[case.block_tables[s, 0], 0], "fp16")
        for hq in range(case.num_q_heads):
            assert np.array_equal(out[s, hq], v[hq // G])


def test_softmax_is_max_subtracted():
    # Step 3 subtracts the maximum before exponentiating; without it these
    # scores overflow float64
    p = oracle.attention_weights(np.array([1000.0, 1001.0, -np.inf]))
    assert np.allclose(p, [1 / (1 + math.e), math.e / (1 + math.e), 0.0], atol=1e-15, rtol=0)


def test_weights_sum_to_one():
    rng = np.random.default_rng(3)
    p = oracle.attention_weights(rng.standard_normal((5, 37)) * 10)
    assert np.allclose(p.sum(axis=-1), 1.0, atol=1e-14)
    assert np.all(p >= 0)


def test_gqa_equals_mha_with_replicated_kv():
    case = _small_case(seed=12, Hq=6, Hkv=2)
    G = case.group
    gqa = _run(case)
    kc = np.repeat(case.key_cache, G, axis=2)
    vc = np.repeat(case.value_cache, G, axis=2)
    mha = _run(case, kc, vc)
    # the group is computed as one [G, d] x [d, L] product, MHA row by row:
    # equal up to summation order
    assert np.allclose(gqa, mha, rtol=1e-13, atol=1e-14)


def test_zero_length_gives_zero_output():
    case = _small_case(seed=13)
    case.seq_lens[1] = 0
    out = _run(case)
    assert np.all(out[1] == 0)


def test_pairs_match_full():
    case = _small_case(seed=14)
    full = _run(case)
    pairs = [(0, 0), (1, 3), (2, 2)]
    got = oracle.paged_decode_pairs(case.query, case.key_cache, case.value_cache,
                                    case.block_tables, case.seq_lens, case.block_size,
                                    case.scale, case.dtype, pairs)
    for (s, h), row in zip(pairs, got):
        assert np.allclose(row, full[s, h], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# Split-K combine
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [[0, 37], [0, 5, 37], [0, 1, 2, 30, 37], [0, 16, 32, 37]])
def test_partition_combine_equals_unsplit(cuts):
    rng = np.random.default_rng(len(cuts))
    K = rng.standard_normal((37, 8))
    V = rng.standard_normal((37, 8))
    q = rng.standard_normal(8) * 3
    direct, _ = oracle.single_query_attention(q, K, V, 0.4)
    parts = [oracle.partition_stats(q, K, V, 0.4, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.allclose(oracle.combine_partitions(parts), direct, rtol=1e-13, atol=1e-14)
    # lse is log(sum(exp(scores))) over the range (scalar-loop check)
    for (a, b), (lse, _) in zip(zip(cuts[:-1], cuts[1:]), parts):
        sc = [0.4 * sum(float(q[i]) * float(K[t, i]) for i in range(8)) for t in range(a, b)]
        m = max(sc)
        assert abs(lse - (m + math.log(math.fsum(math.exp(x - m) for x in sc)))) <= 1e-12


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------
def test_reshape_and_cache_round_trip():
    case = _small_case(seed=15, dtype="bf16")
    T, Hkv, d = 11, case.num_kv_heads, case.head_dim
    B = case.block_size
    rng = np.random.default_rng(0)
    key = W.normal_bits((T, Hkv, d), "bf16", 1, 1)
    val = W.normal_bits((T, Hkv, d), "bf16", 1, 2)
    slots = rng.choice(case.num_blocks * B, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    kc, vc = oracle.reshape_and_cache(key, val, case.key_cache, case.value_cache, slots, B)
    flat_k = kc.reshape(-1, Hkv, d)
    flat_v = vc.reshape(-1, Hkv, d)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(flat_k[s], key[i]) and np.array_equal(flat_v[s], val[i])
    untouched = np.ones(case.num_blocks * B, bool)
    untouched[slots[slots >= 0]] = False
    assert np.array_equal(flat_k[untouched], case.key_cache.reshape(-1, Hkv, d)[untouched])
    assert np.array_equal(flat_v[untouched], case.value_cache.reshape(-1, Hkv, d)[untouched])
    # the inputs were not modified
    assert not np.array_equal(kc, case.key_cache)


def test_write_then_read_through_table():
    # the decode step's write lands where a gather through the table finds it
    case = _small_case(seed=16)
    kc, vc = oracle.reshape_and_cache(case.new_key, case.new_value, case.key_cache,
                                      case.value_cache, case.slot_mapping, case.block_size)
    for s in range(case.num_seqs):
        L = int(case.seq_lens[s])
        K = oracle.gather_kv(kc, case.block_tables[s], L, case.block_size)
        assert np.array_equal(K[L - 1], case.new_key[s])


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------
def test_to_float64_known_patterns():
    assert oracle.to_float64(np.array([0x3F80, 0xC040, 0x0001, 0x7F80], np.uint16), "bf16").tolist() == \
        [1.0, -3.0, 2.0 ** -133, math.inf]
    assert oracle.to_float64(np.array([0x3C00, 0xC200, 0x0001, 0x7C00], np.uint16), "fp16").tolist() == \
        [1.0, -3.0, 2.0 ** -24, math.inf]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_round_to_dtype_idempotent_on_all_patterns(dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = oracle.to_float64(bits, dtype)
    fin = np.isfinite(x) & ~((x == 0) & (np.signbit(x)))
    assert np.array_equal(oracle.round_to_dtype(x[fin], dtype), bits[fin])


def test_round_to_bf16_ties_and_no_double_rounding():
    one = 1.0
    vals = np.array([one + 2 ** -8, one + 3 * 2 ** -8, one + 2 ** -8 + 2 ** -30, -(one + 2 ** -8 + 2 ** -30)])
    assert oracle.round_to_dtype(vals, "bf16").tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF81]


def test_generator_bf16_rounding_matches_oracle_rounding():
    # two independent RNE implementations (integer trick vs scale-and-round)
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    assert np.array_equal(W.f32_to_bits(x, "bf16"), oracle.round_to_dtype(x.astype(np.float64), "bf16"))
    assert np.array_equal(W.f32_to_bits(x, "fp16"), oracle.round_to_dtype(x.astype(np.float64), "fp16"))
