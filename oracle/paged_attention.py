"""Plain float64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline and ``--impl reference`` legs) may import this
module; the CUDA library never does, and the two share no code.

What it computes (sources are the three pages on PagedAttention):

* The output is exactly standard attention over the sequence's tokens in
  logical order ("Paged Attention > The PagedAttention Algorithm",
  Standard Attention vs PagedAttention, the softmax(QK^T/sqrt(d_k))V
  equation; "PagedAttention by hand", Why divide memory into physical blocks?:
  the numerical output equals standard attention). So the oracle is that
  definition, written out: gather the blocks through the table into a
  contiguous K/V (the gather-then-attend reference, In[16]), then a
  max-subtracted softmax (PagedAttention by hand, Forward pass, Step 3) and a
  probability-weighted sum of V (Step 4).
* Logical token ``t`` lives in physical block ``table[t // B]`` at offset
  ``t % B`` (The PagedAttention Algorithm, opening: the example that maps a
  token of a sequence to an offset inside a numbered physical block).
* Only tokens ``t < seq_len`` exist; slots past it are never read
  (PagedAttention by hand, Step 2: bound the loop so invalid slots are never
  touched).
* Inputs are fp16/bf16 bit patterns, widened exactly to float64.
* The cache write puts token ``i``'s K/V row into ``slot_mapping[i]``
  (= physical block * B + offset; negative = skip), the step vLLM performs
  before attention (PagedAttention by hand, Setup, Step 1, and the Code
  section).
* Split-K: attention over a token range gives (log-sum-exp, normalised
  output); ranges combine by log-sum-exp weights. This is the running
  max / running sum of the online softmax (The PagedAttention Algorithm,
  Optimized CUDA Kernels) applied to whole ranges.

Every function is pinned by ``tests/test_oracle.py`` against something other
than itself: the printed worked example, closed forms, brute force with scalar
loops, and the invariants the pages state.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------
def to_float64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of fp16 / bf16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest fp16 / bf16 value (ties to even).

    Returns uint16 bit patterns. bf16 rounding is done in one step from
    float64 (no double rounding through float32): the value is scaled by a
    power of two so the 8 significant bits become the integer part, rounded
    half-to-even, and scaled back.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    ax = np.abs(np.where(finite, x, 0.0))
    _, e = np.frexp(ax)                        # ax = m * 2**e, m in [0.5, 1)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))  # quantum: 8 significant bits
    r = np.round(ax / q) * q                    # np.round: half to even
    out[...] = np.where(finite, np.copysign(r, x), x)
    return (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Address translation and gather
# ---------------------------------------------------------------------------
def gather_kv(cache: np.ndarray, table_row: Sequence[int], seq_len: int,
              block_size: int) -> np.ndarray:
    """Contiguous ``[seq_len, ...]`` rows of one sequence, in logical order.

    Uses ceil(seq_len / B) table entries; the last block contributes only its
    first ``seq_len - j*B`` rows (The PagedAttention Algorithm, In[16]).
    Entries past the last used block are never looked at.
    """
    B = block_size
    n = (seq_len + B - 1) // B
    parts = []
    for j in range(n):
        phys = int(table_row[j])
        take = min(B, seq_len - j * B)
        parts.append(cache[phys, :take])
    if not parts:
        return cache[:0, 0]
    return np.concatenate(parts, axis=0)


# ---------------------------------------------------------------------------
# Attention for one query vector
# ---------------------------------------------------------------------------
def attention_weights(scores: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis (PagedAttention by hand, Step 3).

    Entries equal to -inf get weight exactly 0 (Step 2's masking).
    """
    s = np.asarray(scores, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def single_query_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                           scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """softmax(scale * K q) V for one query (standard attention, n x d_k keys).

    ``q`` is ``[d]`` or ``[G, d]`` (a group of query heads sharing K/V);
    returns ``(out, probs)``. With no tokens the output is zero.
    """
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[:-1] + (V.shape[-1],)), np.zeros(q.shape[:-1] + (0,))
    scores = (q @ K.T) * scale
    p = attention_weights(scores)
    return p @ V, p


# ---------------------------------------------------------------------------
# Paged decode
# ---------------------------------------------------------------------------
def paged_decode(query, key_cache, value_cache, block_tables, seq_lens,
                 block_size: int, scale: float, dtype: str,
                 seqs: Optional[Iterable[int]] = None) -> np.ndarray:
    """Single-query decode attention over a paged KV cache, float64.

    ``query`` [S, Hq, d], caches [NB, B, Hkv, d] (bit patterns of ``dtype``),
    ``block_tables`` [S, MB], ``seq_lens`` [S]. Query head ``hq`` reads kv head
    ``hq // (Hq / Hkv)`` (contiguous groups). Returns float64 [S, Hq, d]
    (rows of sequences not in ``seqs`` are left zero).
    """
    S, Hq, d = query.shape
    Hkv = key_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((S, Hq, d), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        L = int(seq_lens[s])
        K = to_float64(gather_kv(key_cache, block_tables[s], L, block_size), dtype)
        V = to_float64(gather_kv(value_cache, block_tables[s], L, block_size), dtype)
        q = to_float64(query[s], dtype)
        for h in range(Hkv):
            o, _ = single_query_attention(q[h * G:(h + 1) * G], K[:, h, :], V[:, h, :], scale)
            out[s, h * G:(h + 1) * G] = o
    return out


def paged_decode_pairs(query, key_cache, value_cache, block_tables, seq_lens,
                       block_size: int, scale: float, dtype: str,
                       pairs: Iterable[Tuple[int, int]]) -> np.ndarray:
    """The same as :func:`paged_decode` for selected (sequence, query head) pairs.

    Returns float64 [len(pairs), d]; used to check full-size runs one output
    row at a time.
    """
    Hq = query.shape[1]
    Hkv = key_cache.shape[2]
    G = Hq // Hkv
    res = []
    for s, hq in pairs:
        L = int(seq_lens[s])
        h = hq // G
        K = to_float64(gather_kv(key_cache[:, :, h], block_tables[s], L, block_size), dtype)
        V = to_float64(gather_kv(value_cache[:, :, h], block_tables[s], L, block_size), dtype)
        o, _ = single_query_attention(to_float64(query[s, hq], dtype), K, V, scale)
        res.append(o)
    return np.stack(res) if res else np.zeros((0, query.shape[2]))


# ---------------------------------------------------------------------------
# Paged causal prefill (chunked prefill)
# ---------------------------------------------------------------------------
def paged_prefill(query, key_cache, value_cache, block_tables, seq_lens, query_start,
                  block_size: int, scale: float, dtype: str) -> np.ndarray:
    """Causal attention of a chunk of new tokens over a paged cache, float64.

    ``query`` [total_q, Hq, d]: sequence s owns rows query_start[s] ..
    query_start[s+1]-1, its Q_s newest tokens; with L = seq_lens[s] (the
    chunk's K/V already in the cache), query j sits at position L - Q_s + j
    and attends to tokens 0 .. L - Q_s + j ("PagedAttention" glossary, How It
    Works: the blockwise formula with query index i, read token by token so
    every token up to i counts once and none after it). Returns float64
    [total_q, Hq, d].
    """
    total_q, Hq, d = query.shape
    Hkv = key_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((total_q, Hq, d), dtype=np.float64)
    for s in range(len(seq_lens)):
        L = int(seq_lens[s])
        q0, q1 = int(query_start[s]), int(query_start[s + 1])
        Q = q1 - q0
        K = to_float64(gather_kv(key_cache, block_tables[s], L, block_size), dtype)
        V = to_float64(gather_kv(value_cache, block_tables[s], L, block_size), dtype)
        for j in range(Q):
            p = L - Q + j
            q = to_float64(query[q0 + j], dtype)
            for h in range(Hkv):
                o, _ = single_query_attention(q[h * G:(h + 1) * G], K[:p + 1, h, :], V[:p + 1, h, :], scale)
                out[q0 + j, h * G:(h + 1) * G] = o
    return out


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------
def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                      block_size: int, in_place: bool = False):
    """Write token i's K/V rows ([Hkv, d]) into slot ``slot_mapping[i]``.

    slot = physical block * B + offset; a negative slot means "no write".
    Bit copy, element by element. Returns the (possibly copied) caches.
    """
    kc = key_cache if in_place else key_cache.copy()
    vc = value_cache if in_place else value_cache.copy()
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        kc[blk, off] = key[i]
        vc[blk, off] = value[i]
    return kc, vc


# ---------------------------------------------------------------------------
# Split-K over token ranges
# ---------------------------------------------------------------------------
def partition_stats(q, K, V, scale: float, lo: int, hi: int):
    """(log-sum-exp of scaled scores, softmax-normalised output) over tokens [lo, hi)."""
    q = np.asarray(q, dtype=np.float64)
    s = (K[lo:hi] @ q) * scale
    m = np.max(s)
    w = np.exp(s - m)
    l = np.sum(w)
    return m + math.log(l), (w @ V[lo:hi]) / l


def combine_partitions(parts):
    """Merge (lse_p, o_p) pairs: o = sum_p exp(lse_p - M) o_p / sum_p exp(lse_p - M)."""
    lse = np.array([p[0] for p in parts], dtype=np.float64)
    M = np.max(lse)
    w = np.exp(lse - M)
    o = sum(wi * np.asarray(p[1], dtype=np.float64) for wi, p in zip(w, parts))
    return o / np.sum(w)
