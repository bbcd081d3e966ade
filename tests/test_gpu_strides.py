"""Paged pools passed as views into larger allocations (include/csa.h, "Pool
strides"): every call gives bit-identical results to the same call on dense
pools -- page strides (pools of several layers side by side) and row strides
(several fields per row)."""

import numpy as np
import pytest
import torch

from workloads import BLOCK, make_workload, random_selection, spec_for
import oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefill_csa_compress_gb300 as csa  # noqa: E402
from prefill_csa_compress_gb300.pipeline import CsaStep  # noqa: E402

DEV = torch.device("cuda:0")


def _page_strided(pool, fill=7):
    """The same pool inside a [pages, 3, 128, ...] allocation (layer 1 of 3)."""
    big = torch.full((pool.shape[0], 3) + tuple(pool.shape[1:]), fill, dtype=pool.dtype,
                     device=pool.device)
    big[:, 1] = pool
    return big[:, 1]


def _row_strided(pool, fill=7):
    """The same pool with two fields per row ([pages, 128, 2, width], field 0)."""
    big = torch.full(tuple(pool.shape[:2]) + (2,) + tuple(pool.shape[2:]), fill, dtype=pool.dtype,
                     device=pool.device)
    big[:, :, 0] = pool
    return big[:, :, 0]


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_on_strided_pools(prefill):
    spec = spec_for("serving_decode", topk=256, seed=101)
    wl = make_workload(spec)
    t = wl.to(DEV)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 3).to(DEV)
    fn = csa.csa_sparse_attn_prefill if prefill else csa.csa_sparse_attn_decode
    outs = []
    for kv, cmp in ((t["kv_pool"], t["cmp_pool"]),
                    (_page_strided(t["kv_pool"]), _row_strided(t["cmp_pool"])),
                    (_row_strided(t["kv_pool"]), _page_strided(t["cmp_pool"]))):
        out = torch.zeros_like(t["q"])
        lse = torch.zeros(t["q"].shape[:2], dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        fn(q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=sel, kv_pool=kv,
           kv_block_table=t["kv_table"], kv_len=t["kv_len"], cmp_pool=cmp,
           cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"], ratio=spec.ratio, out=out, lse=lse,
           sink=t["sink"], rope_cos=t["rope_cos"], rope_sin=t["rope_sin"], status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append((out.cpu(), lse.cpu()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("mode", [csa.CSA_MODE_DECODE, csa.CSA_MODE_PREFILL])
def test_index_on_strided_pools(mode):
    spec = spec_for("serving_decode", seed=102)
    wl = make_workload(spec)
    t = wl.to(DEV)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    res = []
    for keys, scales in ((t["idx_pool"], t["idx_scale"]),
                         (_page_strided(t["idx_pool"]), _page_strided(t["idx_scale"])),
                         (_row_strided(t["idx_pool"]), t["idx_scale"])):
        idx = torch.full((spec.n_rows, spec.topk), -7, dtype=torch.int32, device=DEV)
        sc = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        csa.csa_index_topk(q_idx=t["q_idx"], weights=t["idx_w"], row_req=t["row_req"],
                           row_pos=t["row_pos"], n_cmp=t["n_cmp"], ratio=spec.ratio,
                           idx_pool=keys, idx_scale_pool=scales, cmp_block_table=t["cmp_table"],
                           topk=spec.topk, topk_idx=idx, scores=sc, rope_cos=t["rope_cos"],
                           rope_sin=t["rope_sin"], mode=mode, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append((idx.cpu(), sc.cpu()))
    for i, s_ in res[1:]:
        assert torch.equal(i, res[0][0])
        assert torch.equal(torch.nan_to_num(s_, nan=1e30), torch.nan_to_num(res[0][1], nan=1e30))


def test_reindex_on_strided_keys():
    spec = spec_for("serving_decode", seed=103, topk=64)
    wl = make_workload(spec)
    t = wl.to(DEV)
    n_cand = 32
    cand = torch.full((spec.n_rows, n_cand), -1, dtype=torch.int32, device=DEV)
    base = dict(q_idx=t["q_idx"], weights=t["idx_w"], row_req=t["row_req"], row_pos=t["row_pos"],
                n_cmp=t["n_cmp"], ratio=spec.ratio, cmp_block_table=t["cmp_table"],
                topk=spec.topk, rope_cos=t["rope_cos"], rope_sin=t["rope_sin"])
    lvl = torch.empty((spec.n_rows, spec.topk), dtype=torch.int32, device=DEV)
    csa.csa_index_topk(idx_pool=t["idx_pool"], idx_scale_pool=t["idx_scale"], topk_idx=lvl,
                       cand_out=cand, **base)
    res = []
    for keys, scales in ((t["idx_pool"], t["idx_scale"]),
                         (_row_strided(t["idx_pool"]), _page_strided(t["idx_scale"]))):
        idx = torch.full((spec.n_rows, spec.topk), -7, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        csa.csa_index_topk(idx_pool=keys, idx_scale_pool=scales, topk_idx=idx, cand_in=cand,
                           status=st, **base)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append(idx.cpu())
    assert torch.equal(res[0], res[1])


@pytest.mark.parametrize("n_rows", [12, 600])  # short chunks (fused kernel), long (GEMM + pool)
def test_compress_into_strided_pools(n_rows):
    rng = np.random.default_rng(104 + n_rows)
    ratio, dx = 4, 128
    positions = torch.arange(n_rows, dtype=torch.int32, device=DEV) + 3
    row_req = torch.zeros(n_rows, dtype=torch.int32, device=DEV)
    x = torch.from_numpy(rng.standard_normal((n_rows, dx)).astype(np.float32)).bfloat16().to(DEV)
    table = torch.tensor([[2, 0, 3, 1, 5, 4]], dtype=torch.int32, device=DEV)
    from workloads import rope_tables
    cos, sin = rope_tables(4096)
    res = {}
    for d, out in ((512, "bf16"), (128, "int8")):
        kv = torch.from_numpy(rng.standard_normal((n_rows, d)).astype(np.float32)).bfloat16().to(DEV)
        w = torch.from_numpy((rng.standard_normal((dx, d)) / np.sqrt(dx)).astype(np.float32))
        w = w.bfloat16().to(DEV)
        ape = torch.from_numpy(rng.standard_normal((ratio, d)).astype(np.float32)).to(DEV)
        got = []
        for layout in ("dense", "page", "row"):
            cmp_pool = torch.zeros((6, BLOCK, d), dtype=torch.bfloat16, device=DEV)
            idx_pool = torch.zeros((6, BLOCK, d), dtype=torch.int8, device=DEV)
            idx_scale = torch.zeros((6, BLOCK), dtype=torch.float32, device=DEV)
            if layout == "page":
                cmp_pool, idx_pool, idx_scale = (_page_strided(cmp_pool, 0),
                                                 _page_strided(idx_pool, 0),
                                                 _page_strided(idx_scale, 0))
            elif layout == "row":
                cmp_pool, idx_pool = _row_strided(cmp_pool, 0), _row_strided(idx_pool, 0)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            csa.csa_compress(x=x, kv=kv, w_gate=w, ape=ape, ratio=ratio, positions=positions,
                             row_req=row_req, block_table=table, out=out, cmp_pool=cmp_pool,
                             idx_pool=idx_pool, idx_scale_pool=idx_scale, rotate=out == "int8",
                             rope_cos=cos.to(DEV), rope_sin=sin.to(DEV), status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            got.append((cmp_pool.cpu().clone(), idx_pool.cpu().clone(), idx_scale.cpu().clone()))
        for g in got[1:]:
            for a_, b_ in zip(g, got[0]):
                assert torch.equal(a_, b_), (d, out)
        res[out] = got[0]
    assert res["bf16"][0].abs().sum() > 0 and res["int8"][1].abs().sum() > 0
