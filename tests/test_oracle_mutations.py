"""The oracle's pins catch plausible mistakes.

Each mutation below plants one mistake in the oracle (on the CPU, through
monkeypatch, for the duration of one test): a dropped scale, a softmax without
the max subtraction, query heads mapped to the wrong kv head, the last block
read whole, one block too few, the keys used as values, a wrong split-K
combine, the slot decoded the wrong way round, a wrong bf16 widening, a causal
limit one token too short or too long, positions counted from the chunk start.
With any one of them in place, at least one pin of ``test_oracle.py`` /
``test_oracle_prefill.py`` must fail; with none, all of them pass.
"""
import numpy as np
import pytest

import oracle
import oracle.paged_attention as PA
import test_oracle as T
import test_oracle_prefill as TP

_orig = {name: getattr(PA, name) for name in
         ("single_query_attention", "attention_weights", "gather_kv", "combine_partitions",
          "reshape_and_cache", "to_float64", "paged_decode", "paged_prefill")}

# the pins, with one representative parameter set each
PINS = [
    (T.test_worked_example_output, {"dtype": "fp16"}),
    (T.test_worked_example_output, {"dtype": "bf16"}),
    (T.test_worked_example_scores_and_probs, {}),
    (T.test_step2_masking_gives_zero_weight, {}),
    (T.test_two_token_closed_form, {"scale": 0.125}),
    (T.test_uniform_scores_average_values, {}),
    (T.test_brute_force_random, {"B": 2, "Hq": 4, "Hkv": 2, "d": 8, "dtype": "bf16"}),
    (T.test_brute_force_boundary_lengths, {"lens": [1, 3, 4, 5]}),
    (T.test_demo_shape_scattered_blocks, {}),
    (T.test_placement_independence, {}),
    (T.test_block_size_invariance, {}),
    (T.test_unused_slots_are_never_read, {}),
    (T.test_seq_len_one_returns_v_exactly, {}),
    (T.test_softmax_is_max_subtracted, {}),
    (T.test_weights_sum_to_one, {}),
    (T.test_gqa_equals_mha_with_replicated_kv, {}),
    (T.test_partition_combine_equals_unsplit, {"cuts": [0, 5, 37]}),
    (T.test_reshape_and_cache_round_trip, {}),
    (T.test_write_then_read_through_table, {}),
    (T.test_to_float64_known_patterns, {}),
    (TP.test_single_new_token_is_decode, {}),
    (TP.test_brute_force_causal, {"B": 4, "qlens": [3, 5, 1]}),
    (TP.test_later_tokens_do_not_change_earlier_queries, {}),
    (TP.test_whole_prompt_chunk_equals_decode_at_every_length, {}),
]


def _failures():
    failed = []
    for f, kw in PINS:
        try:
            with np.errstate(all="ignore"):
                f(**kw)
        except Exception:  # an assertion, or a shape error the mistake causes
            failed.append(f.__name__)
    return failed


# ---- the mutants ------------------------------------------------------------
def _no_scale(q, K, V, scale):
    return _orig["single_query_attention"](q, K, V, 1.0)


def _no_max_subtraction(scores):
    e = np.exp(np.asarray(scores, dtype=np.float64))
    return e / np.sum(e, axis=-1, keepdims=True)


def _keys_as_values(q, K, V, scale):
    return _orig["single_query_attention"](q, K, K, scale)


def _whole_last_block(cache, table_row, seq_len, block_size):
    n = (seq_len + block_size - 1) // block_size
    parts = [cache[int(table_row[j]), :block_size] for j in range(n)]
    return np.concatenate(parts, axis=0) if parts else cache[:0, 0]


def _one_block_short(cache, table_row, seq_len, block_size):
    n = seq_len // block_size
    parts = [cache[int(table_row[j]), :min(block_size, seq_len - j * block_size)] for j in range(n)]
    return np.concatenate(parts, axis=0) if parts else cache[:0, 0]


def _plain_average_combine(parts):
    return sum(np.asarray(p[1], dtype=np.float64) for p in parts) / len(parts)


def _slot_swapped(key, value, key_cache, value_cache, slot_mapping, block_size, in_place=False):
    kc = key_cache if in_place else key_cache.copy()
    vc = value_cache if in_place else value_cache.copy()
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        off, blk = divmod(int(slot), block_size)  # wrong way round
        if blk < kc.shape[0] and off < kc.shape[1]:
            kc[blk, off] = key[i]
            vc[blk, off] = value[i]
    return kc, vc


def _bf16_wrong_widening(bits, dtype):
    if dtype == "bf16":
        bits = np.asarray(bits, dtype=np.uint16)
        return (bits.astype(np.uint32) << 15).view(np.float32).astype(np.float64)
    return _orig["to_float64"](bits, dtype)


def _interleaved_heads(query, key_cache, value_cache, block_tables, seq_lens, block_size, scale,
                       dtype, seqs=None):
    S, Hq, d = query.shape
    Hkv = key_cache.shape[2]
    out = np.zeros((S, Hq, d))
    for s in (range(S) if seqs is None else seqs):
        L = int(seq_lens[s])
        K = PA.to_float64(PA.gather_kv(key_cache, block_tables[s], L, block_size), dtype)
        V = PA.to_float64(PA.gather_kv(value_cache, block_tables[s], L, block_size), dtype)
        q = PA.to_float64(query[s], dtype)
        for h in range(Hkv):  # query head hq read kv head hq % Hkv
            o, _ = PA.single_query_attention(q[h::Hkv], K[:, h, :], V[:, h, :], scale)
            out[s, h::Hkv] = o
    return out


def _prefill_variant(limit):
    """paged_prefill with query j seeing tokens [0, limit(L, Q, j)) instead of [0, L - Q + j]."""
    def f(query, key_cache, value_cache, block_tables, seq_lens, query_start, block_size, scale,
          dtype):
        total_q, Hq, d = query.shape
        Hkv = key_cache.shape[2]
        G = Hq // Hkv
        out = np.zeros((total_q, Hq, d))
        for s in range(len(seq_lens)):
            L = int(seq_lens[s])
            q0, q1 = int(query_start[s]), int(query_start[s + 1])
            Q = q1 - q0
            K = PA.to_float64(PA.gather_kv(key_cache, block_tables[s], L, block_size), dtype)
            V = PA.to_float64(PA.gather_kv(value_cache, block_tables[s], L, block_size), dtype)
            for j in range(Q):
                n = max(0, min(L, limit(L, Q, j)))
                q = PA.to_float64(query[q0 + j], dtype)
                for h in range(Hkv):
                    o, _ = PA.single_query_attention(q[h * G:(h + 1) * G], K[:n, h, :],
                                                     V[:n, h, :], scale)
                    out[q0 + j, h * G:(h + 1) * G] = o
        return out
    return f


MUTANTS = {
    "scale dropped": ("single_query_attention", _no_scale),
    "softmax without the max subtraction": ("attention_weights", _no_max_subtraction),
    "keys used as values": ("single_query_attention", _keys_as_values),
    "last block read whole": ("gather_kv", _whole_last_block),
    "one block too few": ("gather_kv", _one_block_short),
    "split-K parts averaged": ("combine_partitions", _plain_average_combine),
    "slot decoded the wrong way round": ("reshape_and_cache", _slot_swapped),
    "bf16 widened by 15 bits": ("to_float64", _bf16_wrong_widening),
    "query heads interleaved over kv heads": ("paged_decode", _interleaved_heads),
    "causal limit one token short": ("paged_prefill", _prefill_variant(lambda L, Q, j: L - Q + j)),
    "causal limit one token long": ("paged_prefill", _prefill_variant(lambda L, Q, j: L - Q + j + 2)),
    "positions counted from the chunk start": ("paged_prefill", _prefill_variant(lambda L, Q, j: j + 1)),
    "whole context visible": ("paged_prefill", _prefill_variant(lambda L, Q, j: L)),
}


def test_the_pins_pass_on_the_oracle_as_it_is():
    assert _failures() == []


@pytest.mark.parametrize("name", list(MUTANTS))
def test_a_planted_mistake_fails_a_pin(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(PA, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    failed = _failures()
    assert failed, f"no pin catches: {name}"
