"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out as a paged KV cache:
it holds none of the attention arithmetic. Both the CPU oracle's tests and the
GPU path's tests and benchmark take their inputs from here, so the two sides
always see the same bits.

Layouts follow "Paged Attention > The PagedAttention Algorithm" (Standard
Attention vs PagedAttention, In[16]):

* ``key_cache`` / ``value_cache``: ``[num_blocks, block_size, num_kv_heads, head_dim]``
* ``block_tables``: ``[num_seqs, max_blocks_per_seq]`` int32 physical block ids
* ``seq_lens``: ``[num_seqs]`` int32
* ``query``: ``[num_seqs, num_q_heads, head_dim]`` (one decode token per sequence)

Element data are 16-bit floats stored as ``uint16`` bit patterns (fp16 or
bf16), rounded to nearest-even from float32 N(0, 1) draws.

Recipe (one ``numpy.random.default_rng`` stream per purpose, all from ``seed``):
sequence lengths are uniform integers over an inclusive range; the physical
pool holds 1.2x the blocks the sequences need (the tiny case: exactly 64); a
random permutation of the pool is dealt out in order, so each sequence owns a
random, unordered set of blocks ("PagedAttention by hand", Step 1: the table
[2, 0, 1]); table entries past a sequence's last block are random in-range ids
that must never be read. The shared-prefix case draws each group's 1024-token
prefix once and points all 8 sequences of the group at the same physical
blocks (a reference count of 8), so it needs no copy-on-write.
"""
from __future__ import annotations

import concurrent.futures as _fut
import dataclasses
import os
from typing import Optional

import numpy as np

DTYPES = ("fp16", "bf16")
_CHUNK = 1 << 22  # elements per independently seeded chunk of a big tensor


# ---------------------------------------------------------------------------
# 16-bit encodings of float32 draws (input preparation, not method arithmetic)
# ---------------------------------------------------------------------------
def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16 or bf16 (nearest-even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        b = x.view(np.uint32)
        nan = (b & 0x7FFFFFFF) > 0x7F800000
        r = (b >> 16) & np.uint32(1)
        out = ((b + np.uint32(0x7FFF) + r) >> 16).astype(np.uint16)
        if nan.any():
            out[nan] = ((b[nan] >> 16) | 0x40).astype(np.uint16)
        return out
    raise ValueError(f"unknown dtype {dtype!r}")


def nan_bits(dtype: str) -> int:
    """A quiet-NaN bit pattern in the given 16-bit format (used to poison memory)."""
    return {"fp16": 0x7E00, "bf16": 0x7FC0}[dtype]


def inf_bits(dtype: str) -> int:
    return {"fp16": 0x7C00, "bf16": 0x7F80}[dtype]


def _fill_chunk(out_flat, lo, hi, seed, stream_id, k, dtype):
    rng = np.random.default_rng([seed, stream_id, k])
    out_flat[lo:hi] = f32_to_bits(rng.standard_normal(hi - lo, dtype=np.float32), dtype)


def normal_bits(shape, dtype: str, seed: int, stream_id: int,
                threads: Optional[int] = None) -> np.ndarray:
    """N(0,1) draws of ``shape`` rounded to ``dtype``; returns uint16 bits.

    The tensor is cut into fixed chunks, chunk ``k`` seeded by
    ``(seed, stream_id, k)``, so the result does not depend on how many
    threads fill it.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    if nchunks <= 1 or threads <= 1:
        for k in range(nchunks):
            _fill_chunk(out, k * _CHUNK, min(n, (k + 1) * _CHUNK), seed, stream_id, k, dtype)
    else:
        with _fut.ThreadPoolExecutor(max_workers=threads) as ex:
            futs = [ex.submit(_fill_chunk, out, k * _CHUNK, min(n, (k + 1) * _CHUNK),
                              seed, stream_id, k, dtype) for k in range(nchunks)]
            for f in futs:
                f.result()
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# Decode cases
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeCase:
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    partition_tokens: int  # 0 = library's choice
    query: np.ndarray          # uint16 [S, Hq, d]
    key_cache: np.ndarray      # uint16 [NB, B, Hkv, d]
    value_cache: np.ndarray    # uint16 [NB, B, Hkv, d]
    block_tables: np.ndarray   # int32 [S, MB]
    seq_lens: np.ndarray       # int32 [S]
    # the decode step's newly produced token (position seq_len-1 of each
    # sequence), written into the cache before attention runs
    new_key: np.ndarray        # uint16 [S, Hkv, d]
    new_value: np.ndarray      # uint16 [S, Hkv, d]
    slot_mapping: np.ndarray   # int64 [S]; -1 = no write for that sequence

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes(self) -> int:
        """K+V bytes that exist for the sequences (no tail-of-block slots)."""
        return int(2 * self.seq_lens.astype(np.int64).sum() * self.num_kv_heads * self.head_dim * 2)

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct valid slots (shared blocks counted once)."""
        seen = {}
        B = self.block_size
        for s in range(self.num_seqs):
            L = int(self.seq_lens[s])
            nb = (L + B - 1) // B
            for j in range(nb):
                phys = int(self.block_tables[s, j])
                seen[phys] = max(seen.get(phys, 0), min(B, L - j * B))
        return int(2 * sum(seen.values()) * self.num_kv_heads * self.head_dim * 2)

    def algorithmic_bytes(self) -> int:
        """Bytes one decode call must move (K/V rows, table entries, lengths, q, out)."""
        B = self.block_size
        L = self.seq_lens.astype(np.int64)
        nblk = (L + B - 1) // B
        e = 2
        return int(self.kv_bytes() + 4 * nblk.sum() + 4 * self.num_seqs
                   + 2 * self.num_seqs * self.num_q_heads * self.head_dim * e)

    def cache_write_bytes(self) -> int:
        """Bytes the cache write moves: read new K and V rows, write them to the cache."""
        n = int((self.slot_mapping >= 0).sum())
        return 4 * n * self.num_kv_heads * self.head_dim * 2 + 8 * self.num_seqs


def _slot_of_last_token(block_tables, seq_lens, block_size):
    S = len(seq_lens)
    slots = np.full(S, -1, dtype=np.int64)
    for s in range(S):
        L = int(seq_lens[s])
        if L > 0:
            t = L - 1
            slots[s] = int(block_tables[s, t // block_size]) * block_size + t % block_size
    return slots


def random_case(*, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                len_range, dtype, seed=0, pool="1.2x", scale=None,
                partition_tokens=0, max_blocks_per_seq=None, name="random",
                seq_lens=None, threads=None) -> DecodeCase:
    """A decode batch with random lengths and randomly placed physical blocks.

    ``pool`` is ``"1.2x"`` (1.2 times the blocks needed, rounded up) or an
    integer pool size (the tiny case deals ``rng.permutation(64)``).
    """
    S, B = num_seqs, block_size
    rng = np.random.default_rng([seed, 1])
    lo, hi = len_range
    if seq_lens is None:
        seq_lens = rng.integers(lo, hi + 1, size=S).astype(np.int32)
    else:
        seq_lens = np.asarray(seq_lens, dtype=np.int32)
    nblk = (seq_lens.astype(np.int64) + B - 1) // B
    need = int(nblk.sum())
    if pool == "1.2x":
        NB = max(1, int(np.ceil(1.2 * need)))
    else:
        NB = int(pool)
        if NB < need:
            raise ValueError("pool too small")
    MB = max_blocks_per_seq if max_blocks_per_seq is not None else max(1, (hi + B - 1) // B)
    perm = rng.permutation(NB).astype(np.int32)
    tables = rng.integers(0, NB, size=(S, MB)).astype(np.int32)  # junk tail
    pos = 0
    for s in range(S):
        n = int(nblk[s])
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    query = normal_bits((S, num_q_heads, head_dim), dtype, seed, 2, threads)
    kc = normal_bits((NB, B, num_kv_heads, head_dim), dtype, seed, 3, threads)
    vc = normal_bits((NB, B, num_kv_heads, head_dim), dtype, seed, 4, threads)
    nk = normal_bits((S, num_kv_heads, head_dim), dtype, seed, 5, threads)
    nv = normal_bits((S, num_kv_heads, head_dim), dtype, seed, 6, threads)
    if scale is None:
        scale = 1.0 / float(np.sqrt(head_dim))
    return DecodeCase(name, dtype, S, num_q_heads, num_kv_heads, head_dim, B, NB, MB,
                      float(scale), partition_tokens, query, kc, vc, tables, seq_lens,
                      nk, nv, _slot_of_last_token(tables, seq_lens, B))


def shared_prefix_case(*, block_size, groups=32, per_group=8, prefix=1024,
                       suffix_range=(0, 512), num_heads=32, head_dim=128,
                       dtype="fp16", seed=0, name=None, threads=None) -> DecodeCase:
    """Groups of sequences sharing a prefix of whole blocks (same physical ids).

    The logical K/V of every prefix and suffix is drawn independently of
    ``block_size``; only the placement into the pool depends on it, so the
    same logical cache can be compared across block sizes.
    """
    B = block_size
    if prefix % B:
        raise ValueError("prefix must be whole blocks")
    S = groups * per_group
    H, d = num_heads, head_dim
    rng = np.random.default_rng([seed, 11])
    suf = rng.integers(suffix_range[0], suffix_range[1] + 1, size=S).astype(np.int64)
    seq_lens = (prefix + suf).astype(np.int32)
    pre_k = normal_bits((groups, prefix, H, d), dtype, seed, 12, threads)
    pre_v = normal_bits((groups, prefix, H, d), dtype, seed, 13, threads)
    tot_suf = int(suf.sum())
    suf_k = normal_bits((max(tot_suf, 1), H, d), dtype, seed, 14, threads)
    suf_v = normal_bits((max(tot_suf, 1), H, d), dtype, seed, 15, threads)
    query = normal_bits((S, H, d), dtype, seed, 16, threads)
    nk = normal_bits((S, H, d), dtype, seed, 17, threads)
    nv = normal_bits((S, H, d), dtype, seed, 18, threads)

    pre_blocks = prefix // B
    suf_blocks = (suf + B - 1) // B
    need = groups * pre_blocks + int(suf_blocks.sum())
    NB = int(np.ceil(1.2 * need))
    prng = np.random.default_rng([seed, 19, B])
    perm = prng.permutation(NB).astype(np.int32)
    MB = pre_blocks + (suffix_range[1] + B - 1) // B
    tables = prng.integers(0, NB, size=(S, MB)).astype(np.int32)
    kc = np.zeros((NB, B, H, d), dtype=np.uint16)
    vc = np.zeros((NB, B, H, d), dtype=np.uint16)
    pos = 0
    for g in range(groups):
        ids = perm[pos:pos + pre_blocks]
        pos += pre_blocks
        kc[ids] = pre_k[g].reshape(pre_blocks, B, H, d)
        vc[ids] = pre_v[g].reshape(pre_blocks, B, H, d)
        for i in range(per_group):
            tables[g * per_group + i, :pre_blocks] = ids
    off = 0
    for s in range(S):
        n = int(suf[s])
        nb = int(suf_blocks[s])
        ids = perm[pos:pos + nb]
        pos += nb
        tables[s, pre_blocks:pre_blocks + nb] = ids
        for j in range(nb):
            m = min(B, n - j * B)
            kc[ids[j], :m] = suf_k[off + j * B: off + j * B + m]
            vc[ids[j], :m] = suf_v[off + j * B: off + j * B + m]
        off += n
    # the new token is the last suffix token; a sequence without a suffix would
    # write into a shared prefix block (a copy-on-write case), so it skips
    slots = _slot_of_last_token(tables, seq_lens, B)
    slots[suf == 0] = -1
    return DecodeCase(name or f"shared_prefix_B{B}", dtype, S, H, H, d, B, NB, MB,
                      1.0 / float(np.sqrt(d)), 0, query, kc, vc, tables, seq_lens,
                      nk, nv, slots)


# The five workloads, named for what they are.
WORKLOADS = {
    "tiny": dict(num_seqs=4, num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                 len_range=(1, 128), dtype="fp16", pool=64),
    "llama2_7b_mha": dict(num_seqs=64, num_q_heads=32, num_kv_heads=32, head_dim=128,
                          block_size=16, len_range=(512, 2048), dtype="fp16"),
    "llama3_8b_gqa": dict(num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, len_range=(1024, 8192), dtype="bf16"),
    "long_context_splitk": dict(num_seqs=8, num_q_heads=64, num_kv_heads=8, head_dim=128,
                                block_size=16, len_range=(32768, 131072), dtype="bf16",
                                partition_tokens=512),
}
SHARED_PREFIX_BLOCK_SIZES = (1, 8, 16, 32, 64)


def make_workload(name: str, seed: int = 0, block_size: Optional[int] = None,
                  threads=None, num_seqs: Optional[int] = None) -> DecodeCase:
    """Build one of the named workloads (``shared_prefix`` takes ``block_size``).

    ``num_seqs`` shrinks the batch (same per-sequence recipe), for profiling
    captures that must stay small.
    """
    if name == "shared_prefix":
        kw = {} if num_seqs is None else {"groups": max(1, num_seqs // 8)}
        return shared_prefix_case(block_size=block_size or 16, seed=seed, threads=threads, **kw)
    kw = dict(WORKLOADS[name])
    if num_seqs is not None:
        kw["num_seqs"] = num_seqs
    return random_case(seed=seed, name=name, threads=threads, **kw)


def poison_unused(case: DecodeCase, bits: int) -> None:
    """Overwrite every slot no sequence can read (pool blocks not in any table
    prefix, and tail slots of each last block) with ``bits`` in place."""
    B = case.block_size
    used = np.zeros((case.num_blocks, B), dtype=bool)
    for s in range(case.num_seqs):
        L = int(case.seq_lens[s])
        for j in range((L + B - 1) // B):
            used[int(case.block_tables[s, j]), :min(B, L - j * B)] = True
    case.key_cache[~used] = bits
    case.value_cache[~used] = bits
