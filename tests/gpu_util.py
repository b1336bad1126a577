"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
import paged_kv_cache_305_gb300 as pa

TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}
# max |GPU - float64 oracle| for decode (fp16/bf16 inputs, fp32 accumulation)
ATOL = 2e-3


def dev_bits(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(TORCH_DTYPE[dtype])


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceCase:
    """A workloads.DecodeCase resident on the GPU."""

    def __init__(self, case, device="cuda"):
        self.case = case
        dt = case.dtype
        self.query = dev_bits(case.query, dt, device)
        self.key_cache = dev_bits(case.key_cache, dt, device)
        self.value_cache = dev_bits(case.value_cache, dt, device)
        self.block_tables = torch.from_numpy(case.block_tables).to(device)
        self.seq_lens = torch.from_numpy(case.seq_lens).to(device)
        self.new_key = dev_bits(case.new_key, dt, device)
        self.new_value = dev_bits(case.new_value, dt, device)
        self.slot_mapping = torch.from_numpy(case.slot_mapping).to(device)
        self.out = torch.empty_like(self.query)
        self.out32 = torch.empty(self.query.shape, dtype=torch.float32, device=device)
        self.partition_tokens = case.partition_tokens
        self.workspace = pa.alloc_workspace(self.query, self.key_cache, self.block_tables,
                                            case.partition_tokens)

    def write_new_tokens(self):
        pa.reshape_and_cache(self.new_key, self.new_value, self.key_cache, self.value_cache,
                             self.slot_mapping)

    def decode(self, partition_tokens=None, workspace=None, out_f32=False):
        """Run pa_decode; returns ``out`` (input dtype) or ``out32`` (fp32)."""
        pt = self.partition_tokens if partition_tokens is None else partition_tokens
        ws = self.workspace if partition_tokens is None else workspace
        if partition_tokens is not None and ws is None:
            ws = pa.alloc_workspace(self.query, self.key_cache, self.block_tables, pt)
        out = self.out32 if out_f32 else self.out
        pa.decode(out, self.query, self.key_cache, self.value_cache, self.block_tables,
                  self.seq_lens, self.case.scale, pt, ws)
        return out

    def step(self):
        """One decode step: write the new token's K/V, then attend over the sequence."""
        self.write_new_tokens()
        return self.decode()


def oracle_after_write(case):
    """Oracle caches after the step's cache write (host copies)."""
    return oracle.reshape_and_cache(case.new_key, case.new_value, case.key_cache,
                                    case.value_cache, case.slot_mapping, case.block_size)


def check_parity(out16: np.ndarray, out32: np.ndarray, ref: np.ndarray, dtype: str,
                 what: str = "") -> float:
    """The two-part parity bar for decode.

    1. The fp32 result is within ATOL of the float64 oracle.
    2. The 16-bit output is exactly the nearest-even rounding of that fp32
       result (so its distance from the oracle is the fp32 error plus at most
       half a unit in the last place of the 16-bit type).
    Returns the fp32 error.
    """
    o32 = np.asarray(out32, dtype=np.float64)
    assert np.all(np.isfinite(o32)), f"{what}: non-finite output"
    diff = np.abs(o32 - ref)
    err = float(np.max(diff)) if ref.size else 0.0
    if err > ATOL:
        where = np.unravel_index(int(np.argmax(diff)), diff.shape)
        rows = np.argwhere(diff.reshape(diff.shape[0], -1).max(axis=1) > ATOL).ravel()
        raise AssertionError(f"{what}: max |fp32 - oracle| = {err} at {tuple(int(x) for x in where)}; "
                             f"{len(rows)} rows above tolerance, first {rows[:12].tolist()}")
    rounded = oracle.round_to_dtype(o32, dtype)
    bad = int(np.sum(rounded != out16))
    assert bad == 0, f"{what}: {bad} 16-bit outputs differ from the rounding of the fp32 result"
    return err


def max_err(got_bits: np.ndarray, ref: np.ndarray, dtype: str) -> float:
    got = oracle.to_float64(got_bits, dtype)
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(np.max(np.abs(got - ref))) if ref.size else 0.0
