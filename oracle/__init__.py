"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under
``paged_kv_cache_305_gb300/`` never imports it and shares no code with it.

Every function here is a plain float64 restatement of what the source pages
define; see ``paged_attention.py`` for the citations and the pins that check
it in ``tests/test_oracle.py``.
"""
from .paged_attention import (  # noqa: F401
    to_float64,
    gather_kv,
    attention_weights,
    single_query_attention,
    paged_decode,
    paged_decode_pairs,
    paged_prefill,
    reshape_and_cache,
    partition_stats,
    combine_partitions,
    round_to_dtype,
)
