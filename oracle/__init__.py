"""CPU oracle for chunked-prefill causal attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never does.
"""

from .attention import (  # noqa: F401
    BLOCK_SIZE,
    attention_rows,
    causal_attention_probs,
    causal_chunk_attention,
    chunk_flops,
    default_scale,
    gather_paged,
    kv_append,
    merge_partials,
    mixed_batch_attention,
    split_key_range_attention,
)
