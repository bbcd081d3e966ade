"""CPU oracle for compressed sparse attention — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library.
"""

from .csa_oracle import (  # noqa: F401
    BLOCK,
    LowBitPool,
    as_f64,
    bf16_round,
    cache_rows,
    compress,
    compress_stateful,
    dequant_fp4,
    dequant_mxfp8,
    e2m1_decode,
    e4m3_decode,
    e8m0_decode,
    index_scores,
    pack_nibbles,
    page_rows,
    quantize_fp4_e4m3,
    quantize_fp4_e8m0,
    quantize_int8,
    quantize_mxfp8,
    round_e2m1,
    round_e4m3,
    rope_rotate,
    select_blocks,
    sparse_attention,
    topk_in_blocks,
    topk_select,
    unpack_nibbles,
    visible_count,
    window_positions,
)
