"""KV-memory waste of paged vs contiguous allocation on a synthetic serving trace.

The pages' headline measurement: pre-reserving a contiguous max-length chunk
per request wastes most of the KV memory (60-80 % in the "PagedAttention"
glossary, Why It Exists), while paged allocation wastes at most B - 1 slots
per sequence ("PagedAttention by hand", waste table: ~15 slots at B = 16).

`simulate` admits requests with random prompt and output lengths, decodes
them token by token, and at every step measures
  * paged: slots actually held by the library's native block manager
    (pa_bm_*: on-demand blocks, freed when a request finishes), and
  * contiguous: max_len slots per live request,
against the tokens really stored. Lengths are drawn from a seeded NumPy
generator: prompts uniform, outputs geometric (most answers short, a long
tail), capped so prompt + output <= max_len.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .pagedattn import BlockManager


@dataclasses.dataclass
class WasteResult:
    block_size: int
    max_len: int
    steps: int
    used_token_steps: int        # sum over steps of tokens stored
    paged_slot_steps: int        # sum over steps of slots held by the block manager
    contiguous_slot_steps: int   # sum over steps of max_len per live request
    max_paged_waste_per_seq: int

    @property
    def paged_waste(self) -> float:
        return 1.0 - self.used_token_steps / self.paged_slot_steps

    @property
    def contiguous_waste(self) -> float:
        return 1.0 - self.used_token_steps / self.contiguous_slot_steps


def simulate(block_size: int = 16, max_len: int = 2048, concurrent: int = 64,
             requests: int = 512, prompt_range=(16, 512), mean_output: float = 200.0,
             seed: int = 0, trace=None) -> WasteResult:
    """Run the trace; if `trace` is a list, the stored lengths of the live
    requests are appended to it at every step."""
    rng = np.random.default_rng(seed)
    B = block_size
    mb = (max_len + B - 1) // B
    bm = BlockManager(concurrent * mb, B, mb)
    prompts = rng.integers(prompt_range[0], prompt_range[1] + 1, size=requests)
    outputs = np.minimum(rng.geometric(1.0 / mean_output, size=requests), max_len - prompts)
    pending = list(range(requests))[::-1]
    live = {}  # seq id -> [tokens stored, tokens to reach]
    used = paged = contig = steps = 0
    worst = 0
    while pending or live:
        while pending and len(live) < concurrent:
            r = pending.pop()
            sid = bm.new_sequence()
            bm.append([(sid, int(prompts[r]))])
            live[sid] = [int(prompts[r]), int(prompts[r] + outputs[r])]
        reqs = [(sid, 1) for sid, (n, end) in live.items() if n < end]
        if reqs:
            bm.append(reqs)
            for sid, _ in reqs:
                live[sid][0] += 1
        stored = sum(v[0] for v in live.values())
        if trace is not None:
            trace.append([v[0] for v in live.values()])
        held = (bm.block_size * (concurrent * mb - bm.num_free_blocks()))
        used += stored
        paged += held
        contig += max_len * len(live)
        steps += 1
        worst = max(worst, max((-v[0]) % B for v in live.values()))
        for sid in [s for s, (n, end) in live.items() if n >= end]:
            bm.free_sequence(sid)
            del live[sid]
    bm.close()
    return WasteResult(B, max_len, steps, used, paged, contig, worst)
