"""CPU oracle (fp64) for quantized-KV decode attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
it. It shares no code with the GPU library and imports nothing from it.
"""
from .qda_oracle import (  # noqa: F401
    DTYPES,
    attention,
    attention_blocked,
    attention_head_compat,
    attention_packed_compat,
    attention_two_pass_blocked,
    cache_append,
    attention_head,
    attention_packed,
    attention_packed_multi,
    bits16,
    dequantize,
    from_bits16,
    pack,
    qgemv,
    quantize,
    quantize_cache,
    round_to,
    seq_row_offsets,
    unit_rows,
    unpack,
    visible_rows,
)
