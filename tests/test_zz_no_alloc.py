"""csa_index_topk_noalloc against csa_index_topk, through the C ABI.

The no-allocation variant serves callers that may not hand the library any
device memory (an engine plugin whose memory is planned ahead, or a decode loop
that must not call the CUDA allocator); it keeps its score scratch in an
array inside the library.  It must select exactly what the workspace-based
entry point selects, call after call, although the array keeps the previous
call's contents.  This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from parity import SCORE_REL  # noqa: E402
from prefill_csa_compress_gb300 import _binding as B  # noqa: E402
from workloads import make_workload, spec_for  # noqa: E402

DEV = torch.device("cuda:0")


def _args(t, topk, topk_idx, topk_score, workspace=None, ws_bytes=0):
    a = B.IndexArgs()
    a.struct_size = ctypes.sizeof(B.IndexArgs)
    a.n_rows, a.n_heads, a.head_dim = (int(x) for x in t["q_idx"].shape)
    a.ratio, a.topk, a.relu, a.mode = 2, topk, 1, B.CSA_MODE_DECODE
    a.q_idx, a.weights = t["q_idx"].data_ptr(), t["idx_w"].data_ptr()
    a.row_req, a.row_pos, a.n_cmp = (t[k].data_ptr() for k in ("row_req", "row_pos", "n_cmp"))
    a.idx_pool, a.idx_scale_pool = t["idx_pool"].data_ptr(), t["idx_scale"].data_ptr()
    a.cmp_block_table = t["cmp_table"].data_ptr()
    a.n_req, a.max_blocks = (int(x) for x in t["cmp_table"].shape)
    a.n_blocks = int(t["idx_pool"].shape[0])
    a.rope_cos, a.rope_sin = t["rope_cos"].data_ptr(), t["rope_sin"].data_ptr()
    a.rope_cap = int(t["rope_cos"].shape[0])
    a.topk_idx, a.topk_score = topk_idx.data_ptr(), topk_score.data_ptr()
    a.workspace, a.workspace_bytes = workspace, ws_bytes
    return a


# Calls in a row over the shared scratch array: the later calls see fewer
# entries per row (and a different row pitch) than the first, so leftover
# scores past a row's visible count are there to be misread if the kernel
# ever read them.
_CALLS = [
    ("serving_decode", dict(seed=61)),
    ("tiny_decode", dict(seed=62)),
    ("serving_decode", dict(ctx=[900, 300, 2000, 129], seed=63)),
]


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row():
    L = B.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for name, over in _CALLS:
        spec = spec_for(name, **over)
        t = make_workload(spec).to(DEV)
        k = spec.topk
        ref_idx = torch.full((spec.n_rows, k), -7, dtype=torch.int32, device=DEV)
        ref_sc = torch.zeros((spec.n_rows, k), dtype=torch.float32, device=DEV)
        q = _args(t, k, ref_idx, ref_sc)
        assert L.csa_index_topk(ctypes.byref(q), None) == B.CSA_OK  # size query
        ws = torch.empty(max(int(q.workspace_bytes), 256), dtype=torch.uint8, device=DEV)
        a = _args(t, k, ref_idx, ref_sc, ws.data_ptr(), ws.numel())
        assert L.csa_index_topk(ctypes.byref(a), stream) == B.CSA_OK
        got_idx = torch.full((spec.n_rows, k), -7, dtype=torch.int32, device=DEV)
        got_sc = torch.zeros((spec.n_rows, k), dtype=torch.float32, device=DEV)
        n = _args(t, k, got_idx, got_sc)
        assert L.csa_index_topk_noalloc(ctypes.byref(n), stream) == B.CSA_OK
        torch.cuda.synchronize()
        assert torch.equal(got_idx, ref_idx), name
        tol = SCORE_REL * ref_sc.abs() + 1e-30
        fin = torch.isfinite(ref_sc)
        assert torch.equal(fin, torch.isfinite(got_sc))
        assert bool(((got_sc - ref_sc).abs()[fin] <= tol[fin]).all())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = B.lib()
    spec = spec_for("serving_decode")
    t = make_workload(spec).to(DEV)
    idx = torch.empty((spec.n_rows, spec.topk), dtype=torch.int32, device=DEV)
    sc = torch.empty((spec.n_rows, spec.topk), dtype=torch.float32, device=DEV)
    a = _args(t, spec.topk, idx, sc)
    a.max_blocks = 65  # rows of 8320 entries: more than one CTA's select handles
    assert L.csa_index_topk_noalloc(ctypes.byref(a), None) == B.CSA_ERR_UNSUPPORTED
    a = _args(t, spec.topk, idx, sc)
    a.n_rows = 300  # 300 x 4096 scores: more than the 2^20-entry scratch
    assert L.csa_index_topk_noalloc(ctypes.byref(a), None) == B.CSA_ERR_UNSUPPORTED
