"""fp64 CPU oracle for the attention hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package; the library never does.
"""

from .attention import (  # noqa: F401
    admissible_keys,
    attention,
    attention_backward,
    attention_fp8,
    attention_fp8_head,
    attention_backward_head,
    attention_backward_rows,
    attention_head,
    backward_delta,
    chunk_partials,
    combine,
    compositions,
    decode,
    decode_paged,
    paged_rows,
    dequantize_blocks,
    e4m3_values,
    online_attention_head,
    online_merge_scores,
    quantize_e4m3_blocks,
    round_to_e4m3,
    shard_partials_head,
)
