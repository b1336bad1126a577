"""Python binding of libpagedattn.so (ctypes; argument marshalling only).

Every step of the computation runs in the library's CUDA kernels. PyTorch is
used for device memory and streams only: tensors are passed by
``data_ptr()`` and work is enqueued on the current CUDA stream of the
tensors' device. If the library is missing this module raises; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedattn.so")

PA_FLOAT16, PA_BFLOAT16, PA_FLOAT32 = 0, 1, 2
_DTYPES = {torch.float16: PA_FLOAT16, torch.bfloat16: PA_BFLOAT16}
EXPORTED = ("pa_reshape_and_cache", "pa_decode_workspace_bytes", "pa_decode",
            "pa_last_error", "pa_bad_index_count", "pa_decode_no_alloc",
            "pa_decode_no_alloc_scratch_bytes", "pa_copy_blocks", "pa_bm_create",
            "pa_bm_destroy", "pa_bm_new_sequence", "pa_bm_fork", "pa_bm_free_sequence",
            "pa_bm_append", "pa_bm_block_tables", "pa_bm_num_free_blocks", "pa_bm_ref_count",
            "pa_decode_append", "pa_prefill", "pa_wait_timeout_count",
            "pa_testing_prefill_stalled", "pa_prefill_workspace_bytes",
            "pa_decode_partition_tokens")
PA_ERR_CAPACITY = -5

_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"pagedattn error {code}: {msg}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpagedattn.so and declare the C signatures (raises if absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built: run `python -m paged_kv_cache_305_gb300.build` "
            "(needs nvcc); there is no CPU fallback")
    L = ctypes.CDLL(path)
    vp, i32, i64p, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    L.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, i64p, i32, i32, i32, i32, i32, i32, vp]
    L.pa_reshape_and_cache.restype = i32
    L.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.pa_decode_workspace_bytes.restype = sz
    L.pa_decode_partition_tokens.argtypes = [i32, i32, i32]
    L.pa_decode_partition_tokens.restype = i32
    L.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                            i32, i32, i32, i32, i32, vp, sz, vp]
    L.pa_decode.restype = i32
    L.pa_last_error.argtypes = []
    L.pa_last_error.restype = ctypes.c_char_p
    L.pa_bad_index_count.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
    L.pa_bad_index_count.restype = i32
    L.pa_wait_timeout_count.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
    L.pa_wait_timeout_count.restype = i32
    L.pa_decode_no_alloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     ctypes.c_float, i32, i32, i32, i32, i32, vp]
    L.pa_decode_no_alloc.restype = i32
    L.pa_decode_no_alloc_scratch_bytes.argtypes = []
    L.pa_decode_no_alloc_scratch_bytes.restype = sz
    L.pa_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                   ctypes.c_float, i32, i32, i32, i32, i32, vp, sz, vp]
    L.pa_decode_append.restype = i32
    L.pa_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                             i32, i32, i32, i32, i32, vp, sz, vp]
    L.pa_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.pa_prefill_workspace_bytes.restype = sz
    L.pa_prefill.restype = i32
    L.pa_testing_prefill_stalled.argtypes = L.pa_prefill.argtypes
    L.pa_testing_prefill_stalled.restype = i32
    L.pa_copy_blocks.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    L.pa_copy_blocks.restype = i32
    ip = ctypes.POINTER(ctypes.c_int)
    L.pa_bm_create.argtypes = [i32, i32, i32, ctypes.POINTER(vp)]
    L.pa_bm_create.restype = i32
    L.pa_bm_destroy.argtypes = [vp]
    L.pa_bm_destroy.restype = None
    L.pa_bm_new_sequence.argtypes = [vp, ip]
    L.pa_bm_new_sequence.restype = i32
    L.pa_bm_fork.argtypes = [vp, i32, ip]
    L.pa_bm_fork.restype = i32
    L.pa_bm_free_sequence.argtypes = [vp, i32]
    L.pa_bm_free_sequence.restype = i32
    L.pa_bm_append.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, ip]
    L.pa_bm_append.restype = i32
    L.pa_bm_block_tables.argtypes = [vp, vp, i32, vp, vp]
    L.pa_bm_block_tables.restype = i32
    L.pa_bm_num_free_blocks.argtypes = [vp, ip]
    L.pa_bm_num_free_blocks.restype = i32
    L.pa_bm_ref_count.argtypes = [vp, i32, ip]
    L.pa_bm_ref_count.restype = i32
    _lib = L
    return L


def last_error() -> str:
    return load_library().pa_last_error().decode()


def _check(rc: int) -> None:
    if rc != 0:
        raise PagedAttnError(rc, last_error())


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype} (float16 or bfloat16)")
    return _DTYPES[t.dtype]


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                      value_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Write key/value [T, Hkv, d] rows into the caches [NB, B, Hkv, d] at slot_mapping [T] (int64)."""
    _need(key.is_cuda and key.is_contiguous() and value.is_contiguous()
          and key_cache.is_contiguous() and value_cache.is_contiguous()
          and slot_mapping.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(key.dtype == value.dtype == key_cache.dtype == value_cache.dtype, "dtype mismatch")
    NB, B, Hkv, d = key_cache.shape
    _need(value_cache.shape == key_cache.shape, "key/value cache shape mismatch")
    T = key.shape[0]
    _need(key.shape == (T, Hkv, d) and value.shape == (T, Hkv, d), "key/value shape mismatch")
    _need(slot_mapping.shape == (T,), "slot_mapping shape mismatch")
    L = load_library()
    with torch.cuda.device(key.device):
        _check(L.pa_reshape_and_cache(key.data_ptr(), value.data_ptr(), key_cache.data_ptr(),
                                      value_cache.data_ptr(), slot_mapping.data_ptr(), T, Hkv, d,
                                      B, NB, _dtype_code(key), _stream(key, stream)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                           max_blocks_per_seq: int, block_size: int,
                           partition_tokens: int = 0) -> int:
    return int(load_library().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                        max_blocks_per_seq, block_size,
                                                        partition_tokens))


def decode_partition_tokens(partition_tokens: int, block_size: int,
                            max_blocks_per_seq: int) -> int:
    """The split-K partition length pa_decode resolves these arguments to."""
    rc = load_library().pa_decode_partition_tokens(partition_tokens, block_size,
                                                   max_blocks_per_seq)
    if rc < 0:
        raise PagedAttnError(rc, last_error())
    return int(rc)


def alloc_workspace(query: torch.Tensor, key_cache: torch.Tensor, block_tables: torch.Tensor,
                    partition_tokens: int = 0) -> Optional[torch.Tensor]:
    """Zero-filled workspace for :func:`decode` with these shapes (None if none is needed)."""
    S, Hq, d = query.shape
    n = decode_workspace_bytes(S, Hq, d, block_tables.shape[1], key_cache.shape[1], partition_tokens)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=query.device)


def decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
           value_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
           scale: float, partition_tokens: int = 0,
           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged decode attention into ``out`` [S, Hq, d]; returns ``out``.

    ``query`` [S, Hq, d]; caches [NB, B, Hkv, d]; ``block_tables`` [S, MB]
    int32; ``seq_lens`` [S] int32. ``scale`` multiplies q.K (the caller's
    choice; the library has no default, e.g. 1/sqrt(d) for standard attention). ``out``
    has the query's dtype (rounded result) or float32 (the result before that
    rounding). The workspace, when one is needed, comes from
    :func:`alloc_workspace` (zeroed once, reusable across calls on one stream).
    """
    S, Hq, d = query.shape
    NB, B, Hkv, d2 = key_cache.shape
    _need(d2 == d and value_cache.shape == key_cache.shape, "cache shape mismatch")
    _need(out.shape == query.shape and query.dtype == key_cache.dtype == value_cache.dtype
          and out.dtype in (query.dtype, torch.float32), "out/query/cache dtype or shape mismatch")
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == S and seq_lens.shape == (S,),
          "block_tables/seq_lens shape mismatch")
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    L = load_library()
    with torch.cuda.device(query.device):
        _check(L.pa_decode(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(),
                           value_cache.data_ptr(), block_tables.data_ptr(), seq_lens.data_ptr(),
                           S, Hq, Hkv, d, B, float(scale), block_tables.shape[1], NB,
                           partition_tokens, _dtype_code(query),
                           PA_FLOAT32 if out.dtype == torch.float32 else _dtype_code(query),
                           ws_ptr, ws_bytes,
                           _stream(query, stream)))
    return out


def decode_append(out: torch.Tensor, query: torch.Tensor, new_key: torch.Tensor,
                  new_value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                  block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                  partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """:func:`decode` that also writes each sequence's newest token (position
    seq_lens-1) from ``new_key`` / ``new_value`` [S, Hkv, d] into its slot, in
    the same kernel."""
    S, Hq, d = query.shape
    NB, B, Hkv, d2 = key_cache.shape
    _need(new_key.shape == (S, Hkv, d) and new_value.shape == (S, Hkv, d)
          and new_key.dtype == new_value.dtype == query.dtype, "new_key/new_value shape or dtype mismatch")
    _need(new_key.is_cuda and new_key.is_contiguous() and new_value.is_contiguous(),
          "new_key/new_value must be contiguous CUDA tensors")
    _need(d2 == d and value_cache.shape == key_cache.shape, "cache shape mismatch")
    _need(out.shape == query.shape and query.dtype == key_cache.dtype == value_cache.dtype
          and out.dtype in (query.dtype, torch.float32), "out/query/cache dtype or shape mismatch")
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == S and seq_lens.shape == (S,),
          "block_tables/seq_lens shape mismatch")
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    L = load_library()
    with torch.cuda.device(query.device):
        _check(L.pa_decode_append(out.data_ptr(), query.data_ptr(), new_key.data_ptr(),
                                  new_value.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
                                  block_tables.data_ptr(), seq_lens.data_ptr(), S, Hq, Hkv, d, B,
                                  float(scale), block_tables.shape[1], NB, partition_tokens,
                                  _dtype_code(query),
                                  PA_FLOAT32 if out.dtype == torch.float32 else _dtype_code(query),
                                  ws_ptr, ws_bytes, _stream(query, stream)))
    return out


def prefill_workspace_bytes(num_seqs: int, num_kv_heads: int, head_dim: int,
                            max_blocks_per_seq: int, block_size: int, dtype) -> int:
    """Bytes of the optional :func:`prefill` workspace (an fp16 copy of the value
    rows for bf16 caches; 0 for fp16). ``dtype``: "bf16"/"fp16" or a torch dtype."""
    code = {"fp16": PA_FLOAT16, "bf16": PA_BFLOAT16, torch.float16: PA_FLOAT16,
            torch.bfloat16: PA_BFLOAT16}[dtype]
    return int(load_library().pa_prefill_workspace_bytes(num_seqs, num_kv_heads, head_dim,
                                                         max_blocks_per_seq, block_size, code))


def alloc_prefill_workspace(seq_lens: torch.Tensor, key_cache: torch.Tensor,
                            block_tables: torch.Tensor) -> Optional[torch.Tensor]:
    """Workspace for :func:`prefill` with these shapes (None when it needs none).
    Its contents need no initialisation."""
    NB, B, Hkv, d = key_cache.shape
    n = prefill_workspace_bytes(seq_lens.shape[0], Hkv, d, block_tables.shape[1], B, key_cache.dtype)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=key_cache.device)


def _prefill(entry, out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
            value_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
            query_start: torch.Tensor, max_query_len: int, scale: float,
            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    total_q, Hq, d = query.shape
    NB, B, Hkv, d2 = key_cache.shape
    S = seq_lens.shape[0]
    _need(d2 == d and value_cache.shape == key_cache.shape, "cache shape mismatch")
    _need(out.shape == query.shape and query.dtype == key_cache.dtype == value_cache.dtype
          and out.dtype in (query.dtype, torch.float32), "out/query/cache dtype or shape mismatch")
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32
          and query_start.dtype == torch.int32, "block_tables, seq_lens, query_start must be int32")
    _need(block_tables.shape[0] == S and query_start.shape == (S + 1,), "shape mismatch")
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens, query_start):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    L = load_library()
    with torch.cuda.device(query.device):
        _check(getattr(L, entry)(
            out.data_ptr(), query.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
            block_tables.data_ptr(), seq_lens.data_ptr(), query_start.data_ptr(), S, Hq, Hkv, d, B,
            float(scale), block_tables.shape[1], NB, int(max_query_len), _dtype_code(query),
            PA_FLOAT32 if out.dtype == torch.float32 else _dtype_code(query), ws_ptr, ws_bytes,
            _stream(query, stream)))
    return out


def prefill(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
            value_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
            query_start: torch.Tensor, max_query_len: int, scale: float,
            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal attention of each sequence's newest tokens over the paged cache.

    ``query``/``out`` [total_q, Hq, d]; sequence s owns query rows
    query_start[s] .. query_start[s+1]-1 (int32 [S+1]), its newest tokens,
    whose K/V are already in the cache; ``max_query_len`` bounds the rows per
    sequence. ``workspace`` (optional, :func:`alloc_prefill_workspace`): with
    bf16 caches the value rows are converted to an fp16 copy there and P.V is
    one fp16 product; without it bf16 takes two products.
    """
    return _prefill("pa_prefill", out, query, key_cache, value_cache, block_tables, seq_lens,
                    query_start, max_query_len, scale, workspace, stream)


def testing_prefill_stalled(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, block_tables: torch.Tensor,
                            seq_lens: torch.Tensor, query_start: torch.Tensor, max_query_len: int,
                            scale: float, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Test hook (include/pagedattn_testing.h): :func:`prefill` whose product
    thread waits on a barrier nothing signals, so bounded waits give up and
    the launch winds down; ``out`` is left unwritten."""
    return _prefill("pa_testing_prefill_stalled", out, query, key_cache, value_cache,
                    block_tables, seq_lens, query_start, max_query_len, scale, workspace, stream)


def bad_index_count(clear: bool = False) -> int:
    """Out-of-range indices the kernels skipped on the current device (synchronises)."""
    n = ctypes.c_ulonglong(0)
    _check(load_library().pa_bad_index_count(ctypes.byref(n), int(bool(clear))))
    return int(n.value)


def wait_timeout_count(clear: bool = False) -> int:
    """Bounded in-kernel waits that gave up on the current device (synchronises); 0 when healthy."""
    n = ctypes.c_ulonglong(0)
    _check(load_library().pa_wait_timeout_count(ctypes.byref(n), int(bool(clear))))
    return int(n.value)


def decode_no_alloc(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                    value_cache: torch.Tensor, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, scale: float,
                    partition_tokens: int = 0, stream=None) -> torch.Tensor:
    """:func:`decode` for callers that cannot allocate device memory.

    The split-K scratch is the library's own fixed device array
    (:func:`no_alloc_scratch_bytes` bytes), so no workspace is passed and
    nothing is allocated. Calls that may overlap on the GPU share that array
    and must be serialised by the caller.
    """
    S, Hq, d = query.shape
    NB, B, Hkv, d2 = key_cache.shape
    _need(d2 == d and value_cache.shape == key_cache.shape, "cache shape mismatch")
    _need(out.shape == query.shape and query.dtype == key_cache.dtype == value_cache.dtype
          and out.dtype in (query.dtype, torch.float32), "out/query/cache dtype or shape mismatch")
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == S and seq_lens.shape == (S,),
          "block_tables/seq_lens shape mismatch")
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    L = load_library()
    with torch.cuda.device(query.device):
        _check(L.pa_decode_no_alloc(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(),
                                    value_cache.data_ptr(), block_tables.data_ptr(),
                                    seq_lens.data_ptr(), S, Hq, Hkv, d, B, float(scale),
                                    block_tables.shape[1], NB, partition_tokens,
                                    _dtype_code(query),
                                    PA_FLOAT32 if out.dtype == torch.float32 else _dtype_code(query),
                                    _stream(query, stream)))
    return out


def no_alloc_scratch_bytes() -> int:
    """Bytes of the fixed split-K scratch behind :func:`decode_no_alloc`."""
    return int(load_library().pa_decode_no_alloc_scratch_bytes())


def copy_blocks(key_cache: torch.Tensor, value_cache: torch.Tensor, src: torch.Tensor,
                dst: torch.Tensor, stream=None) -> None:
    """Copy whole blocks src[i] -> dst[i] (int32 CUDA tensors) in both caches."""
    _need(key_cache.is_cuda and key_cache.is_contiguous() and value_cache.is_contiguous(),
          "caches must be contiguous CUDA tensors")
    _need(src.dtype == torch.int32 and dst.dtype == torch.int32 and src.shape == dst.shape
          and src.dim() == 1 and src.is_cuda and dst.is_cuda, "src/dst must be 1-D int32 CUDA tensors")
    NB, B, Hkv, d = key_cache.shape
    L = load_library()
    with torch.cuda.device(key_cache.device):
        _check(L.pa_copy_blocks(key_cache.data_ptr(), value_cache.data_ptr(), src.data_ptr(),
                                dst.data_ptr(), src.numel(), Hkv, d, B, NB, _dtype_code(key_cache),
                                _stream(key_cache, stream)))


class BlockManager:
    """The library's native block manager (host memory; see include/pagedattn.h)."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.pa_bm_create(num_blocks, block_size, max_blocks_per_seq, ctypes.byref(h)))
        self._h = h
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq

    def close(self) -> None:
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_sequence(self) -> int:
        out = ctypes.c_int()
        _check(self._lib.pa_bm_new_sequence(self._h, ctypes.byref(out)))
        return out.value

    def fork(self, parent: int) -> int:
        out = ctypes.c_int()
        _check(self._lib.pa_bm_fork(self._h, parent, ctypes.byref(out)))
        return out.value

    def free_sequence(self, seq_id: int) -> None:
        _check(self._lib.pa_bm_free_sequence(self._h, seq_id))

    def append(self, requests):
        """Slots for new tokens of (seq_id, count) requests and the copy-on-write copies.

        Returns (slot_mapping int64 array, [(src, dst), ...]).
        """
        import numpy as np
        ids = np.array([r[0] for r in requests], dtype=np.int32)
        num = np.array([r[1] for r in requests], dtype=np.int32)
        total = int(num.sum()) if len(num) else 0
        slots = np.zeros(max(total, 1), dtype=np.int64)
        csrc = np.zeros(max(len(ids), 1), dtype=np.int32)
        cdst = np.zeros(max(len(ids), 1), dtype=np.int32)
        nc = ctypes.c_int()
        _check(self._lib.pa_bm_append(self._h, ids.ctypes.data, num.ctypes.data, len(ids),
                                      slots.ctypes.data, total, csrc.ctypes.data, cdst.ctypes.data,
                                      len(ids), ctypes.byref(nc)))
        return slots[:total], [(int(csrc[i]), int(cdst[i])) for i in range(nc.value)]

    def block_tables(self, seq_ids):
        """(int32 [len, max_blocks_per_seq] tables, int32 [len] lengths) of the sequences."""
        import numpy as np
        ids = np.array(seq_ids, dtype=np.int32)
        tables = np.zeros((len(ids), self.max_blocks_per_seq), dtype=np.int32)
        lens = np.zeros(len(ids), dtype=np.int32)
        _check(self._lib.pa_bm_block_tables(self._h, ids.ctypes.data, len(ids), tables.ctypes.data,
                                            lens.ctypes.data))
        return tables, lens

    def num_free_blocks(self) -> int:
        out = ctypes.c_int()
        _check(self._lib.pa_bm_num_free_blocks(self._h, ctypes.byref(out)))
        return out.value

    def ref_count(self, block: int) -> int:
        out = ctypes.c_int()
        _check(self._lib.pa_bm_ref_count(self._h, block, ctypes.byref(out)))
        return out.value
