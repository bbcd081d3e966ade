"""The seeded generator: determinism, shapes and paging structure (no GPU)."""

import numpy as np
import torch

from workloads import BLOCK, make_workload, spec_for


def test_seeded_and_deterministic():
    a = make_workload(spec_for("tiny_decode"))
    b = make_workload(spec_for("tiny_decode"))
    for k in a.t:
        assert torch.equal(a.t[k], b.t[k]), k


def test_serving_decode_layout():
    w = make_workload(spec_for("serving_decode"))
    s = w.spec
    assert w.q.shape == (8, 64, 512) and w.q.dtype == torch.bfloat16
    assert w.q_idx.shape == (8, 64, 128)
    assert w.kv_pool.shape == (256, BLOCK, 512) and w.cmp_pool.shape == (256, BLOCK, 512)
    assert w.idx_pool.dtype == torch.int8 and w.idx_scale.shape == (256, BLOCK)
    assert w.row_pos.tolist() == [8190, 8191, 5998, 5999, 4095, 4096, 2046, 2047]
    assert w.n_cmp.tolist() == [4096, 3000, 2048, 1024]
    # 160 kv pages and 80 cmp pages in use, all distinct
    kv = w.kv_table.numpy()
    cm = w.cmp_table.numpy()
    assert (kv >= 0).sum() == 160 and len(set(kv[kv >= 0].tolist())) == 160
    assert (cm >= 0).sum() == 80 and len(set(cm[cm >= 0].tolist())) == 80
    assert s.topk == 512 and w.rope_cos.shape == (8192, 32)
    # raw rows of the chunk are the window cache rows at those positions
    for t in range(8):
        b, p = int(w.row_req[t]), int(w.row_pos[t])
        assert torch.equal(w.kv_raw[t], w.kv_pool[int(kv[b, p // BLOCK]), p % BLOCK])
    assert np.all(w.idx_pool.numpy() >= -127)


def test_window_only_paging():
    s = spec_for("tiny_decode", ctx=[1024, 700], chunk=[2, 2], kv_pages="window")
    w = make_workload(s)
    kv = w.kv_table.numpy()
    assert kv[0, :6].tolist() == [-1] * 6 and (kv[0, 6:8] >= 0).all()
    assert (kv[1, 4:6] >= 0).all() and kv[1, 3] == -1
