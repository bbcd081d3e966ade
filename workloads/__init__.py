"""Seeded synthetic inputs for compressed sparse attention (CSA).

This module only draws random numbers and lays them out: request contexts,
query rows, paged KV pools with block tables, index keys, compressor weights
and the FP32 half-width RoPE tables.  It holds none of the method's
arithmetic (no compression, scoring, selection or attention) and it is the
only code that the CPU oracle and the CUDA path share.

Value distributions follow the workloads the pages describe (DeepSeek-V4.1
Flash, "Checkpoint shape"; DeepSeek V4-Flash MTP, "Deployment configuration"):
q, q_idx, kv ~ N(0, 1) rounded to BF16; idx_kv uniform integers in
[-127, 127] with an FP32 per-row scale uniform in [1e-3, 1e-2]; index-head
weights N(0, 1)/8; attention sink N(0, 1); softmax scale 1/sqrt(512);
compressor gate weights N(0, 1/D_in); APE N(0, 1).  Block tables are seeded
random permutations of physical 128-row pages.

The RoPE tables are fixture initialisation, as the V4.1 Flash page says of
its table generation ("Serving-owned full RoPE tables"): angle(p, i) =
p * theta**(-2i/rope_dim) with theta = 10000, stored as FP32 cos/sin of
shape [capacity, rope_dim/2].
"""

from .gen import (  # noqa: F401
    BLOCK,
    CONFIGS,
    Workload,
    WorkloadSpec,
    make_workload,
    random_selection,
    reindex_view,
    rope_tables,
    spec_for,
)
