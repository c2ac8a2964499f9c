"""fp64 CPU oracle for GQA attention — test infrastructure, never on the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. See ``gqa_oracle`` for what each
function follows.
"""

from .gqa_oracle import (  # noqa: F401
    NEG_INF,
    TILE_ALL_FUTURE,
    TILE_ALL_PAST,
    TILE_PARTIAL,
    attention,
    attention_q4,
    attention_q8,
    attention_ring,
    attention_rows,
    combine_partials,
    dequantize_q8,
    finalize,
    init_running,
    lse_merge,
    online_softmax_sweep,
    prefill_tile_classes,
    quantize_q4,
    quantize_q8,
    ring_slot,
    ring_visible_tokens,
    ring_write,
    split_bounds,
    split_len,
    split_partials,
    tile_class,
    to_f64,
    visible_count,
)
