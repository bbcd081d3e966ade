"""CPU oracle for compressed sparse attention — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library.
"""

from .csa_oracle import (  # noqa: F401
    BLOCK,
    as_f64,
    bf16_round,
    compress,
    compress_stateful,
    index_scores,
    page_rows,
    quantize_int8,
    rope_rotate,
    select_blocks,
    sparse_attention,
    topk_in_blocks,
    topk_select,
    visible_count,
    window_positions,
)
