"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Small cases span several tiles and ragged tails; the full-size workloads are
checked on sampled rows the oracle computes one by one.  Tolerances are in
``tests/parity.py``.
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import step as OS
from parity import (INT8_FLIP_RATE, LSE_ABS, check_bf16, check_int8_tied, check_scores,
                    check_topk, score_tolerance)
from workloads import BLOCK, make_workload, random_selection, spec_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefill_csa_compress_gb300 as csa  # noqa: E402
import prefill_csa_compress_gb300._binding as B  # noqa: E402
from prefill_csa_compress_gb300.pipeline import CsaStep  # noqa: E402

DEV = torch.device("cuda:0")


_CACHE = {}


def _load(spec):
    key = repr(spec)
    if key not in _CACHE:
        if len(_CACHE) > 2:
            _CACHE.clear()
        _CACHE[key] = make_workload(spec)
    wl = _CACHE[key]
    return wl, wl.to(DEV)


def _status(step):
    return int(step.status.item()) if step.status is not None else 0


def _rope_q(t, row, key="q_idx"):
    p = int(t["row_pos"][row])
    return O.rope_rotate(t[key][row], p, t["rope_cos"], t["rope_sin"])


# ------------------------------------------------------------------ compressor


@pytest.mark.parametrize("name,over", [
    ("chunked_prefill", dict(ctx=[1000], chunk=[1000], seed=31)),       # ragged: 250 groups
    ("chunked_prefill", dict(ctx=[1030, 70], chunk=[1030, 70], ratio=2, seed=32, pad_rows=3)),
    ("chunked_prefill", dict(ctx=[300], chunk=[300], ratio=1, seed=33)),
    # at most 256 rows: both compressors in one fused launch
    ("chunked_prefill", dict(ctx=[203], chunk=[203], seed=34)),
    ("chunked_prefill", dict(ctx=[130, 61], chunk=[130, 61], ratio=1, seed=35, pad_rows=2)),
    ("serving_decode", {}),
    ("stateful_decode", {}),                                            # state rings
    ("hca_prefill", dict(ctx=[700], chunk=[700], seed=61)),             # ratio 128, ragged
    ("hca_decode", {}),                                                 # ratio 128 + ring
    ("chunked_prefill", {}),                                            # full 8192-token chunk
    # overlapping ratio-4 compressors: long chunk, short chunks, chunks that
    # start inside a request (their first window is incomplete), state rings
    ("chunked_prefill", dict(ctx=[1000], chunk=[1000], seed=36, overlap=True)),
    ("chunked_prefill", dict(ctx=[150, 90], chunk=[150, 90], seed=37, overlap=True, pad_rows=2)),
    ("chunked_prefill", dict(ctx=[900, 500], chunk=[601, 298], seed=38, overlap=True)),
    ("stateful_decode", dict(overlap=True)),
    ("stateful_decode", dict(chunk=[37, 6, 3, 1], seed=39, overlap=True)),
    ("chunked_prefill", dict(overlap=True, seed=40)),                   # full 8192-token chunk
])
def test_compress_parity(name, over):
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=spec.mode == "prefill", dense=spec.dense,
                   overlap=spec.overlap)
    step.compress()
    torch.cuda.synchronize()
    assert _status(step) == 0
    trace = {}
    pools, main, idx = OS.compress_step(wl.t, spec, trace=trace)
    table = wl.cmp_table.numpy()
    got_cmp = t["cmp_pool"].cpu()
    got_idx = t["idx_pool"].cpu()
    got_sc = t["idx_scale"].cpu()
    assert (len(main) == len(idx) > 0 or spec.name == "serving_decode" or
            (spec.dense and len(main) > 0 and not idx))
    g_rows, r_rows = [], []
    n_diff = 0
    for b, g, vals in main:
        pg, row = int(table[b, g // BLOCK]), g % BLOCK
        g_rows.append(got_cmp[pg, row].double().numpy())
        r_rows.append(vals)
    for (b, g, codes, scale), rec in zip(idx, trace["idx"]):
        pg, row = int(table[b, g // BLOCK]), g % BLOCK
        n_diff += check_int8_tied(got_idx[pg, row].numpy(), got_sc[pg, row].item(), codes,
                                  np.float32(scale), rec, spec.idx_dim)
    check_bf16(np.stack(g_rows), np.stack(r_rows), "cmp_kv")
    # INT8 codes differ (by one) only at rounding ties, and rarely
    assert n_diff <= INT8_FLIP_RATE * len(idx) * spec.idx_dim + 2, n_diff
    if spec.state:
        # the rings: kv rows exactly, gate scores to FP32 accuracy
        for name in ("state_main",) if spec.dense else ("state_main", "state_idx"):
            got_s = t[name].cpu().double().numpy()
            ref_s = pools[name]
            d = got_s.shape[2] // 2
            assert np.array_equal(got_s[..., :d], ref_s[..., :d]), name
            err = np.abs(got_s[..., d:] - ref_s[..., d:])
            assert np.all(err <= 1e-4 * np.maximum(1.0, np.abs(ref_s[..., d:]))), (name, err.max())
    # entries not written by this step are untouched
    written = {(b, g) for b, g, _ in main}
    ref_pool = wl.cmp_pool
    for b in range(spec.n_req):
        for g in range(0, int(wl.n_cmp[b]), 97):
            if (b, g) not in written:
                pg = int(table[b, g // BLOCK])
                assert torch.equal(got_cmp[pg, g % BLOCK], ref_pool[pg, g % BLOCK])


@pytest.mark.parametrize("n_rows,ratio,dx,d,out,with_gamma", [
    (12, 4, 512, 512, "bf16", False),    # short chunk: fused kernel, 16-column slices
    (12, 2, 192, 512, "bf16", False),    # fused kernel, K = 192
    (600, 2, 192, 512, "bf16", False),   # long chunk: tensor-core GEMM with a 3-chunk K loop
    (12, 4, 128, 128, "int8", True),     # short chunk: fused whole-row kernel with RMSNorm
    (7, 1, 256, 128, "bf16", True),
    (12, 2, 512, 512, "bf16", True),     # RMSNorm over 512 channels: GEMM + pooling kernels
    (600, 4, 512, 512, "int8", True),    # long chunk: tensor-core gate GEMM + pooling kernel
])
def test_compress_direct(n_rows, ratio, dx, d, out, with_gamma):
    """csa_compress called directly: x separate from kv, optional RMSNorm,
    rotation at the group start, BF16 or INT8 output."""
    _compress_direct(n_rows, ratio, dx, d, out, with_gamma)


@pytest.mark.parametrize("n_rows,ratio,dx,d,out,with_gamma", [
    (12, 4, 512, 512, "bf16", False),    # short chunk: gate rows + pooling kernel
    (600, 4, 512, 512, "bf16", False),   # long chunk: tensor-core gate GEMM
    (600, 4, 128, 128, "int8", True),    # rotated INT8 keys with RMSNorm
    (40, 2, 192, 512, "bf16", True),
    (9, 1, 128, 128, "bf16", False),
])
def test_compress_direct_overlap(n_rows, ratio, dx, d, out, with_gamma):
    """The overlapping compressor: each entry pools the previous group's
    tokens too; the chunk's first entries, whose windows start before it,
    are not published."""
    _compress_direct(n_rows, ratio, dx, d, out, with_gamma, overlap=True)


def _compress_direct(n_rows, ratio, dx, d, out, with_gamma, overlap=False):
    rng = np.random.default_rng(n_rows * 7 + ratio + (5 if overlap else 0))
    pos0 = 4 * 37 + 1  # the chunk starts mid-group: its first rows form no group
    positions = np.arange(pos0, pos0 + n_rows, dtype=np.int32)
    row_req = np.zeros(n_rows, np.int32)
    x = torch.from_numpy(rng.standard_normal((n_rows, dx)).astype(np.float32)).bfloat16()
    kv = torch.from_numpy(rng.standard_normal((n_rows, d)).astype(np.float32)).bfloat16()
    w = torch.from_numpy((rng.standard_normal((dx, d)) / np.sqrt(dx)).astype(np.float32)).bfloat16()
    ape = torch.from_numpy(rng.standard_normal((ratio, d)).astype(np.float32))
    gamma = (torch.from_numpy(rng.uniform(0.5, 1.5, d).astype(np.float32)).bfloat16()
             if with_gamma else None)
    from workloads import rope_tables
    cos, sin = rope_tables(4096)
    n_pages = 4
    table = torch.tensor([[2, 0, 3, 1]], dtype=torch.int32)
    cmp_pool = torch.zeros((n_pages, BLOCK, d), dtype=torch.bfloat16, device=DEV)
    idx_pool = torch.zeros((n_pages, BLOCK, d), dtype=torch.int8, device=DEV)
    idx_scale = torch.zeros((n_pages, BLOCK), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.csa_compress(x=x.to(DEV), kv=kv.to(DEV), w_gate=w.to(DEV), ape=ape.to(DEV), ratio=ratio,
                     positions=torch.from_numpy(positions).to(DEV),
                     row_req=torch.from_numpy(row_req).to(DEV), block_table=table.to(DEV),
                     out=out, cmp_pool=cmp_pool, idx_pool=idx_pool, idx_scale_pool=idx_scale,
                     gamma=gamma.to(DEV) if gamma is not None else None, rotate=True,
                     rope_cos=cos.to(DEV), rope_sin=sin.to(DEV), status=status, overlap=overlap)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    trace = []
    ref = O.compress(x, kv, w, ape, ratio, positions, row_req, gamma=gamma, rotate=True,
                     rope_cos=cos, rope_sin=sin, out=out, overlap=overlap, trace=trace)
    first = (pos0 + ratio - 1) // ratio + (1 if overlap else 0)  # first entry with its window here
    assert len(ref) == (pos0 + n_rows) // ratio - first
    got_rows, ref_rows, n_diff = [], [], 0
    for item, rec in zip(ref, trace):
        g = item[1]
        pg, row = int(table[0, g // BLOCK]), g % BLOCK
        if out == "bf16":
            got_rows.append(cmp_pool[pg, row].cpu().double().numpy())
            ref_rows.append(item[2])
        else:
            n_diff += check_int8_tied(idx_pool[pg, row].cpu().numpy(), idx_scale[pg, row].item(),
                                      item[2], np.float32(item[3]), rec, dx)
    if out == "bf16":
        check_bf16(np.stack(got_rows), np.stack(ref_rows), "compressed rows")
    else:
        assert n_diff <= INT8_FLIP_RATE * len(ref) * d + 2, (n_diff, len(ref) * d)


# ------------------------------------------------------------------ indexer


def _stable_topk(scores, k):
    order = np.lexsort((np.arange(len(scores)), -scores.astype(np.float64)))
    return np.sort(order[:k]).astype(np.int32)


def _check_index_rows(wl, t, spec, step, rows, scores_dev):
    torch.cuda.synchronize()
    assert _status(step) == 0
    pools = {"cmp_pool": wl.cmp_pool, "idx_pool": wl.idx_pool, "idx_scale": wl.idx_scale}
    sel = step.topk_idx.cpu().numpy()
    sc_all = scores_dev.cpu().numpy() if scores_dev is not None else None
    n_clear = 0
    for row in rows:
        b = int(wl.row_req[row])
        if b < 0:
            assert np.all(sel[row] == -1)  # untouched padding row (initialised to -1)
            continue
        ref = OS.index_row(wl.t, spec, pools, row)
        V = len(ref)
        keys = O.page_rows(wl.idx_pool, wl.cmp_table[b].numpy(), range(V))
        scl = O.page_rows(wl.idx_scale, wl.cmp_table[b].numpy(), range(V))
        floor = score_tolerance(_rope_q(wl.t, row), O.as_f64(wl.idx_w[row]), keys, scl)
        if sc_all is not None:
            tol = check_scores(sc_all[row, :V], ref, floor)
            # the selection is exactly the (score desc, index asc) top-k of the
            # scores the kernel computed
            mine = _stable_topk(sc_all[row, :V], spec.topk)
            assert np.array_equal(sel[row][:len(mine)], mine)
            assert np.all(sel[row][len(mine):] == -1)
        else:
            tol = np.maximum(1e-4 * np.abs(ref), floor)
        n_clear += check_topk(sel[row], ref, tol, spec.topk)
        # scores reported for the selection match the oracle's
        chosen = sel[row][sel[row] >= 0]
        ts = step.topk_score.cpu().numpy()[row][:len(chosen)]
        assert np.all(np.abs(ts - ref[chosen]) <= np.maximum(1e-4 * np.abs(ref[chosen]),
                                                             floor[chosen]))
    return n_clear


@pytest.mark.parametrize("name,over", [
    ("tiny_decode", {}),
    ("serving_decode", {}),
    ("serving_decode", dict(ctx=[300, 5, 129, 2000], chunk=[3, 1, 2, 40], topk=64, seed=41,
                            pad_rows=2)),
    ("chunked_prefill", dict(ctx=[700], chunk=[700], cmp_init="random", topk=40, seed=42)),
    ("ratio1_decode", dict(ctx=[3000, 2500], chunk=[2, 2], topk=1024, seed=43)),
])
def test_index_topk_parity(name, over):
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=spec.mode == "prefill", compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    _check_index_rows(wl, t, spec, step, range(spec.n_rows), scores)


@pytest.mark.parametrize("name", ["ratio1_decode", "million_decode"])
def test_index_topk_full_size_every_row(name):
    spec = spec_for(name)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.empty((spec.n_rows, n_cap), device=DEV)
    step.index(scores=scores)
    _check_index_rows(wl, t, spec, step, range(spec.n_rows), scores)
    # the workspace path (no caller score buffer) selects the same entries
    sel_a = step.topk_idx.clone()
    step.index()
    torch.cuda.synchronize()
    assert torch.equal(sel_a, step.topk_idx)


@pytest.mark.parametrize("ctx,topk,distinct", [([3000, 2500], 512, 3), ([40000, 30000], 2048, 3),
                                               ([40000, 30000], 2048, 24), ([9000, 8500], 2048, 3)])
def test_index_topk_exact_ties(ctx, topk, distinct):
    # a few distinct key rows under one scale: each query row's scores take
    # `distinct` values, so the cut falls inside a large group of equal scores
    # and the smallest positions of that group must be taken (one CTA per row
    # for 3000 and 9000 entries, rows split over many CTAs for 40000: with 3
    # values the k-th key's first-digit bin is too crowded for the bin path,
    # with 24 it is not, and its equal keys span every slice)
    spec = spec_for("ratio1_decode", ctx=ctx, chunk=[2, 2], topk=topk, seed=44)
    wl = make_workload(spec)
    pick = torch.from_numpy(
        np.random.default_rng(7).integers(0, distinct, size=wl.idx_pool.shape[:2]))
    base = wl.idx_pool[0, :distinct].clone()
    wl.t["idx_pool"] = base[pick].contiguous()
    wl.t["idx_scale"] = torch.full_like(wl.idx_scale, float(wl.idx_scale[0, 0]))
    t = wl.to(DEV)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.empty((spec.n_rows, n_cap), device=DEV)
    step.index(scores=scores)
    _check_index_rows(wl, t, spec, step, range(spec.n_rows), scores)


@pytest.mark.parametrize("four_rows", [False, True])
def test_index_topk_prefill_full_size_sampled(four_rows):
    # the default tiling (rows in pairs) and the four-row one (CSA_MODE_PREFILL)
    spec = spec_for("chunked_prefill", cmp_init="random")
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=True, compress=False)
    if four_rows:
        step.index_mode = B.CSA_MODE_PREFILL
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.empty((spec.n_rows, n_cap), device=DEV)
    step.index(scores=scores)
    _check_index_rows(wl, t, spec, step, [0, 3, 2046, 2047, 2048, 4095, 8191], scores)


# ------------------------------------------------------------------ attention


def _attn_case(spec, sel_seed, prefill, rows=None, use_sink=True, inv_rope_out=False,
               softmax_scale=None, shrink_first=0, sink_values=None):
    if sink_values is not None:
        wl = make_workload(spec)
        wl.t["sink"] = torch.tensor(sink_values, dtype=torch.float32)
        t = wl.to(DEV)
    elif shrink_first:
        # a fresh workload whose first `shrink_first` compressed entries are
        # scaled down 16x: the first candidate tile then has far smaller logits
        # than the later ones and the running maximum must move
        wl = make_workload(spec)
        for b in range(spec.n_req):
            for c in range(shrink_first):
                pg = int(wl.cmp_table[b, c // BLOCK])
                wl.cmp_pool[pg, c % BLOCK] = (wl.cmp_pool[pg, c % BLOCK].float() / 16).bfloat16()
        t = wl.to(DEV)
    else:
        wl, t = _load(spec)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              if int(wl.row_req[i]) >= 0 else 0 for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, sel_seed)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=prefill, compress=False)
    if not use_sink:
        t["sink"] = None
    if inv_rope_out or softmax_scale is not None:
        fn = csa.csa_sparse_attn_prefill if prefill else csa.csa_sparse_attn_decode
        fn(q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=sel.to(DEV),
           kv_pool=t["kv_pool"], kv_block_table=t["kv_table"], kv_len=t["kv_len"],
           cmp_pool=t["cmp_pool"], cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"],
           ratio=spec.ratio, out=step.out, lse=step.lse, sink=t["sink"],
           softmax_scale=softmax_scale, rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
           inv_rope_out=inv_rope_out, status=step.status)
    else:
        step.attention(topk_idx=sel.to(DEV))
    torch.cuda.synchronize()
    assert _status(step) == 0
    out = step.out.cpu().double().numpy()
    lse = step.lse.cpu().numpy()
    pools = {"cmp_pool": wl.cmp_pool}
    rows = range(spec.n_rows) if rows is None else rows
    g, r, gl, rl = [], [], [], []
    for row in rows:
        if int(wl.row_req[row]) < 0:
            assert np.all(out[row] == 0)  # padding rows untouched (zero-initialised)
            continue
        if softmax_scale is None:
            o_ref, l_ref = OS.attention_row(wl.t, spec, pools, row, sel[row].numpy(),
                                            use_sink=use_sink, inv_rope_out=inv_rope_out)
        else:
            b = int(wl.row_req[row])
            o_ref, l_ref = O.sparse_attention(
                wl.q[row], int(wl.row_pos[row]), sel[row].numpy(), wl.kv_pool,
                wl.kv_table[b].numpy(), wl.cmp_pool, wl.cmp_table[b].numpy(),
                wl.sink if use_sink else None, softmax_scale, window=spec.window,
                rope_cos=wl.rope_cos, rope_sin=wl.rope_sin, inv_rope_out=inv_rope_out)
        g.append(out[row])
        r.append(o_ref)
        gl.append(lse[row])
        rl.append(l_ref)
    mag = max(1.0, float(np.max(np.abs(np.stack(r)))) / 2)
    check_bf16(np.stack(g), np.stack(r), "attention out", magnitude=mag)
    assert np.max(np.abs(np.stack(gl) - np.stack(rl))) <= LSE_ABS * max(1.0, np.max(np.abs(rl)))


@pytest.mark.parametrize("prefill", [False, True])
@pytest.mark.parametrize("name,over", [
    ("tiny_decode", {}),
    ("serving_decode", {}),
    ("serving_decode", dict(ctx=[130, 5, 129, 3000], chunk=[3, 5, 2, 7], topk=100, seed=51,
                            pad_rows=2)),
    ("chunked_prefill", dict(ctx=[300], chunk=[300], cmp_init="random", topk=48, seed=52)),
])
def test_attention_parity(name, over, prefill):
    spec = spec_for(name, **over)
    _attn_case(spec, 7, prefill)


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_inverse_rope_output(prefill):
    _attn_case(spec_for("serving_decode", topk=200, seed=54), 11, prefill, inv_rope_out=True)


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_large_logits_move_the_running_max(prefill):
    # logits with a spread of hundreds: the running maximum must move between tiles
    _attn_case(spec_for("chunked_prefill", ctx=[2400], chunk=[5], cmp_init="random", topk=512,
                        seed=55), 12, prefill, softmax_scale=0.15, shrink_first=200)


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_without_sink(prefill):
    _attn_case(spec_for("serving_decode", topk=64, seed=53), 8, prefill, use_sink=False)


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_extreme_sinks(prefill):
    # sinks far above the logits (the sink carries nearly all the weight), far
    # below them, -inf (plain softmax) and ordinary values, head by head
    vals = [40.0, -40.0, -np.inf, 0.0, 12.0, -12.0, 3.0, -3.0] * 8
    _attn_case(spec_for("serving_decode", topk=200, seed=56), 13, prefill, sink_values=vals)


@pytest.mark.parametrize("name", ["ratio1_decode", "million_decode"])
def test_attention_decode_full_size(name):
    _attn_case(spec_for(name), 9, False)


def test_attention_prefill_full_size_sampled():
    spec = spec_for("chunked_prefill", cmp_init="random")
    _attn_case(spec, 10, True, rows=[0, 1, 127, 128, 2047, 4000, 8191])


@pytest.mark.parametrize("ratio,d,out,splits,overlap", [
    (2, 512, "bf16", [[1, 1]] * 6 + [[3, 2], [1, 4], [5, 1]], False),  # decode, then chunks
    (4, 512, "bf16", [[1, 1]] * 7 + [[2, 3], [7, 1], [1, 6]], False),  # chunks longer than the ring
    (4, 128, "int8", [[3, 0], [2, 5], [0, 2], [6, 6]], False),         # idle requests; INT8
    # overlapping windows reach back into the previous group through the ring
    (4, 512, "bf16", [[1, 1]] * 9 + [[2, 3], [7, 1], [1, 6], [10, 11]], True),
    (4, 128, "int8", [[3, 0], [2, 5], [0, 2], [6, 6], [1, 1]], True),
])
def test_compress_state_ring(ratio, d, out, splits, overlap):
    """csa_compress with the recurrent state ring over a chunked stream of two
    requests: the published groups equal the oracle's one-shot compression of
    each request's whole stream, and the ring equals the oracle's ring."""
    rng = np.random.default_rng(ratio * 100 + d + (7 if overlap else 0))
    dx, cap = 256, 2 * ratio if overlap else 4
    lens = [sum(c[b] for c in splits) for b in range(2)]
    n = sum(lens)
    x = torch.from_numpy(rng.standard_normal((n, dx)).astype(np.float32)).bfloat16()
    kv = torch.from_numpy(rng.standard_normal((n, d)).astype(np.float32)).bfloat16()
    w = torch.from_numpy((rng.standard_normal((dx, d)) / np.sqrt(dx)).astype(np.float32)).bfloat16()
    ape = torch.from_numpy(rng.standard_normal((ratio, d)).astype(np.float32))
    from workloads import rope_tables
    cos, sin = rope_tables(4096)
    table = torch.tensor([[3, 1], [0, 2]], dtype=torch.int32)  # 2 requests x 2 pages
    cmp_pool = torch.zeros((4, BLOCK, d), dtype=torch.bfloat16, device=DEV)
    idx_pool = torch.zeros((4, BLOCK, d), dtype=torch.int8, device=DEV)
    idx_scale = torch.zeros((4, BLOCK), dtype=torch.float32, device=DEV)
    state = torch.full((3, cap, 2 * d), 12345.0, dtype=torch.float32, device=DEV)
    state_table = torch.tensor([2, 0], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref_state = np.full((3, cap, 2 * d), 12345.0)
    reqs = [np.arange(0, lens[0]), np.arange(lens[0], n)]
    done = [0, 0]
    for call in splits:
        rows, pos, req = [], [], []
        for b, m in enumerate(call):
            rows += list(reqs[b][done[b]:done[b] + m])
            pos += list(range(done[b], done[b] + m))
            req += [b] * m
            done[b] += m
        idx = np.array(rows)
        kw = dict(rotate=out == "int8", rope_cos=cos, rope_sin=sin, out=out, overlap=overlap)
        O.compress_stateful(x[idx], kv[idx], w, ape, ratio, np.array(pos), np.array(req),
                            ref_state, state_table.numpy(), **kw)
        csa.csa_compress(x=x[idx].to(DEV), kv=kv[idx].to(DEV), w_gate=w.to(DEV), ape=ape.to(DEV),
                         ratio=ratio, positions=torch.tensor(pos, dtype=torch.int32, device=DEV),
                         row_req=torch.tensor(req, dtype=torch.int32, device=DEV),
                         block_table=table.to(DEV), out=out, cmp_pool=cmp_pool, idx_pool=idx_pool,
                         idx_scale_pool=idx_scale, rotate=out == "int8", rope_cos=cos.to(DEV),
                         rope_sin=sin.to(DEV), status=status, state_cache=state,
                         state_block_table=state_table.to(DEV), overlap=overlap)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_rows, ref_rows, n_diff, n_groups = [], [], 0, 0
    for b in range(2):
        i = reqs[b]
        trace = []
        ref = O.compress(x[i], kv[i], w, ape, ratio, np.arange(len(i)), np.zeros(len(i), int),
                         rotate=out == "int8", rope_cos=cos, rope_sin=sin, out=out,
                         overlap=overlap, trace=trace)
        for item, rec in zip(ref, trace):
            g = item[1]
            pg, row = int(table[b, g // BLOCK]), g % BLOCK
            n_groups += 1
            if out == "bf16":
                got_rows.append(cmp_pool[pg, row].cpu().double().numpy())
                ref_rows.append(item[2])
            else:
                n_diff += check_int8_tied(idx_pool[pg, row].cpu().numpy(),
                                          idx_scale[pg, row].item(), item[2],
                                          np.float32(item[3]), rec, dx)
    assert n_groups == sum(l // ratio for l in lens)
    if out == "bf16":
        check_bf16(np.stack(got_rows), np.stack(ref_rows), "compressed rows")
    else:
        assert n_diff <= INT8_FLIP_RATE * n_groups * d + 2, n_diff
    # the ring: kv rows exactly (BF16 -> FP32), gate scores to FP32 accuracy
    got_state = state.cpu().double().numpy()
    assert np.array_equal(got_state[..., :d], ref_state[..., :d])
    err = np.abs(got_state[..., d:] - ref_state[..., d:])
    assert np.all(err <= 1e-4 * np.maximum(1.0, np.abs(ref_state[..., d:]))), err.max()


@pytest.mark.parametrize("name,over", [
    ("serving_decode", {}),
    ("chunked_prefill", dict(ctx=[203], chunk=[203], seed=36)),
    ("chunked_prefill", dict(ctx=[600], chunk=[600], seed=37)),   # long path: four launches
])
def test_compress_pair_equals_two_calls(name, over):
    """csa_compress_pair writes exactly what csa_compress(first) followed by
    csa_compress(second) writes."""
    spec = spec_for(name, **over)
    _, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=spec.mode == "prefill")
    main, keys = step._compress_kw()
    names = ("cmp_pool", "idx_pool", "idx_scale")
    before = {k: t[k].clone() for k in names}
    step.compress()
    torch.cuda.synchronize()
    pair = {k: t[k].clone() for k in names}
    for k in names:
        t[k].copy_(before[k])
    csa.csa_compress(**main)
    csa.csa_compress(**keys)
    torch.cuda.synchronize()
    assert _status(step) == 0
    for k, v in pair.items():
        assert torch.equal(v, t[k]), k


# ------------------------------------------------------------------ whole step


@pytest.mark.parametrize("name,over", [
    ("hca_decode", {}),
    ("hca_prefill", dict(ctx=[1300], chunk=[1300], seed=62)),
    ("hca_decode", dict(lowbit=True, seed=63)),      # FP4 compressed KV, MXFP8 window
])
def test_hca_step(name, over):
    """HCA: ratio-128 compression, then attention over every visible
    compressed entry plus the window, against the oracle's chain."""
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=spec.mode == "prefill", dense=True)
    step.run()
    torch.cuda.synchronize()
    assert _status(step) == 0
    rows = [r for r in range(spec.n_rows) if int(wl.row_req[r]) >= 0]
    if len(rows) > 40:
        rows = rows[:8] + rows[-24:] + list(np.random.default_rng(5).choice(rows, 8, replace=False))
    _, res = OS.full_step(wl.t, spec, rows=rows)
    out = step.out.cpu().double().numpy()
    lse = step.lse.cpu().numpy()
    g = np.stack([out[r] for r in res])
    ref = np.stack([res[r]["out"] for r in res])
    check_bf16(g, ref, "hca out", magnitude=max(1.0, float(np.max(np.abs(ref))) / 2))
    gl = np.stack([lse[r] for r in res])
    rl = np.stack([res[r]["lse"] for r in res])
    assert np.max(np.abs(gl - rl)) <= LSE_ABS * max(1.0, np.max(np.abs(rl)))


@pytest.mark.parametrize("name", ["tiny_decode", "serving_decode", "stateful_decode",
                                  "overlap_decode"])
def test_decode_step_chain(name):
    """compress -> index -> attention on the GPU, against the oracle's own chain."""
    spec = spec_for(name)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, overlap=spec.overlap)
    step.run()
    torch.cuda.synchronize()
    assert _status(step) == 0
    pools, res = OS.full_step(wl.t, spec)
    sel = step.topk_idx.cpu().numpy()
    out = step.out.cpu().double().numpy()
    gpu_idx = t["idx_pool"].cpu()
    same = 0
    for row, rr in res.items():
        b = int(wl.row_req[row])
        V = len(rr["scores"])
        table = wl.cmp_table[b].numpy()
        keys = O.page_rows(pools["idx_pool"], table, range(V))
        scl = O.page_rows(pools["idx_scale"], table, range(V))
        q_rot = _rope_q(wl.t, row)
        w = O.as_f64(wl.idx_w[row])
        floor = score_tolerance(q_rot, w, keys, scl)
        # where the GPU's quantiser rounded a code the other way at a .5 boundary,
        # the score may move by at most scale * sum_h |w_h| * sum_d |q_hd| |dcode_d|
        dcode = np.abs(O.page_rows(gpu_idx, table, range(V)) - keys)
        extra = scl * ((dcode @ np.abs(q_rot).T) @ np.abs(w)) * 1.001
        tol = np.maximum(1e-4 * np.abs(rr["scores"]), floor) + extra
        check_topk(sel[row], rr["scores"], tol, spec.topk)
        if np.array_equal(sel[row], rr["topk"]):
            same += 1
            check_bf16(out[row], rr["out"], f"row {row} out")
    assert same >= len(res) // 2


def test_step_io_staging_matches_plain_step():
    """StepIO packs the per-step inputs and the outputs into single blocks: a
    step fed through one host-to-device copy gives the plain step's results,
    and new inputs written into the host block take effect."""
    from prefill_csa_compress_gb300.pipeline import StepIO

    spec = spec_for("serving_decode", seed=57)
    wl = make_workload(spec)
    names = ["q", "q_idx", "idx_w", "kv_raw", "idx_raw", "row_req", "row_pos", "kv_len", "n_cmp"]
    t1 = wl.to(DEV)
    plain = CsaStep(t1, spec.ratio, spec.topk)
    plain.run()
    t2 = wl.to(DEV)
    io = StepIO(t2, names)
    staged = CsaStep(t2, spec.ratio, spec.topk)
    io.bind_outputs(staged)
    staged.prepare().capture()
    io.h2d()
    staged.replay()
    io.d2h()
    torch.cuda.synchronize()
    n = io.out_bytes
    host = io.host_out[:n]
    out_b = plain.out.numel() * 2
    assert torch.equal(host[:out_b].view(torch.bfloat16).view(plain.out.shape), plain.out.cpu())
    assert torch.equal(staged.topk_idx, plain.topk_idx)
    # a new query written into the host block changes the next step's result
    q_new = io.host_input("q", wl.q)
    q_new.copy_(-wl.q)
    io.h2d()
    staged.replay()
    torch.cuda.synchronize()
    t3 = wl.to(DEV)
    t3["q"] = (-wl.q).to(DEV)
    ref = CsaStep(t3, spec.ratio, spec.topk)
    ref.run()
    torch.cuda.synchronize()
    assert torch.equal(staged.out, ref.out)


def test_step_io_graph_with_late_query_copy():
    """The whole step with its copies as one graph, the query rows copied on
    a side stream that the attention waits for: the plain step's results."""
    from prefill_csa_compress_gb300.pipeline import StepIO

    spec = spec_for("serving_decode", seed=58)
    wl = make_workload(spec)
    names = ["q", "q_idx", "idx_w", "kv_raw", "idx_raw", "row_req", "row_pos", "kv_len", "n_cmp"]
    t1 = wl.to(DEV)
    plain = CsaStep(t1, spec.ratio, spec.topk)
    plain.run()
    t2 = wl.to(DEV)
    io = StepIO(t2, names, late=("q",))
    staged = CsaStep(t2, spec.ratio, spec.topk)
    io.bind_outputs(staged)
    staged.run()
    torch.cuda.synchronize()
    g = io.capture(staged)
    io.host_input("q", wl.q).copy_(2 * wl.q)  # the next step's query
    g.replay()
    torch.cuda.synchronize()
    t3 = wl.to(DEV)
    t3["q"] = (2 * wl.q).to(DEV)
    ref = CsaStep(t3, spec.ratio, spec.topk)
    ref.run()
    torch.cuda.synchronize()
    out_b = ref.out.numel() * 2
    got = io.host_out[:out_b].view(torch.bfloat16).view(ref.out.shape)
    assert torch.equal(got, ref.out.cpu())
    assert torch.equal(staged.topk_idx, plain.topk_idx)



# ------------------------------------------------------------------ head counts


@pytest.mark.parametrize("heads", [16, 96, 128])
@pytest.mark.parametrize("prefill", [False, True])
def test_attention_head_counts(heads, prefill):
    """1 <= heads <= 128: the kernels work in groups of 64 heads; heads past
    the count are padding, computed and never stored."""
    spec = spec_for("serving_decode", heads=heads, topk=256, seed=70 + heads, pad_rows=1)
    _attn_case(spec, 13, prefill)


@pytest.mark.parametrize("idx_heads", [16, 96, 128])
@pytest.mark.parametrize("prefill", [False, True])
def test_index_head_counts(idx_heads, prefill):
    """1 <= index heads <= 128 under both tilings: fewer than 64 are padded with
    zero queries and weights; above 64 a row's score sums its two 64-head
    slots."""
    spec = spec_for("serving_decode", idx_heads=idx_heads, seed=80 + idx_heads, pad_rows=1)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=prefill, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    _check_index_rows(wl, t, spec, step, range(spec.n_rows), scores)


def test_full_size_step_with_128_heads():
    """The whole decode step with 128 query heads and 128 index heads."""
    spec = spec_for("serving_decode", heads=128, idx_heads=128, seed=91)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk)
    step.run()
    torch.cuda.synchronize()
    assert _status(step) == 0
    pools, res = OS.full_step(wl.t, spec)
    sel = step.topk_idx.cpu().numpy()
    out = step.out.cpu().double().numpy()
    g, r = [], []
    for row, rr in res.items():
        b = int(wl.row_req[row])
        V = len(rr["scores"])
        table = wl.cmp_table[b].numpy()
        keys = O.page_rows(pools["idx_pool"], table, range(V))
        scl = O.page_rows(pools["idx_scale"], table, range(V))
        q_rot = _rope_q(wl.t, row)
        w = O.as_f64(wl.idx_w[row])
        tol = np.maximum(1e-4 * np.abs(rr["scores"]), score_tolerance(q_rot, w, keys, scl))
        # keys published differently by the two sides move a score by at most this
        gk = O.page_rows(t["idx_pool"].cpu(), table, range(V))
        gs = O.page_rows(t["idx_scale"].cpu(), table, range(V))
        dk = np.abs(gk * gs[:, None] - keys * scl[:, None])
        tol += ((dk @ np.abs(q_rot).T) @ np.abs(w)) * 1.001
        check_topk(sel[row], rr["scores"], tol, spec.topk)
        g.append(out[row])
        r.append(OS.attention_row(wl.t, spec, pools, row, sel[row])[0])
    check_bf16(np.stack(g), np.stack(r), "out")


# ------------------------------------------------------------------ decode split merge


def _decode_attn_call(spec, t, step, sel, ws=None):
    return csa.csa_sparse_attn_decode(
        q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=sel,
        kv_pool=t["kv_pool"], kv_block_table=t["kv_table"], kv_len=t["kv_len"],
        cmp_pool=t["cmp_pool"], cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"],
        ratio=spec.ratio, out=step.out, lse=step.lse, sink=t["sink"], rope_cos=t["rope_cos"],
        rope_sin=t["rope_sin"], status=step.status, workspace=ws)


@pytest.mark.parametrize("name", ["serving_decode", "million_decode"])
def test_decode_merge_repeats_bit_exactly_on_one_workspace(name):
    # the split counters put themselves back to zero: later calls on the same
    # workspace see the same partials meet and give the same bits
    spec = spec_for(name)
    wl, t = _load(spec)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 21).to(DEV)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    ws = _decode_attn_call(spec, t, step, sel)
    torch.cuda.synchronize()
    assert _status(step) == 0
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    for _ in range(3):
        step.out.zero_()
        ws = _decode_attn_call(spec, t, step, sel, ws)
        torch.cuda.synchronize()
        assert _status(step) == 0
        assert torch.equal(step.out, ref_out) and torch.equal(step.lse, ref_lse)
    # the counters (the last 8 bytes per (row, head group)) read zero again
    assert int(ws[-8 * spec.n_rows:].sum().item()) == 0


def test_decode_merge_counters_not_zero_time_out_loudly():
    # a workspace whose counters do not start at zero: the partials never count
    # up to exactly S, every CTA gives up after its bounded wait, the call raises
    # CSA_DEV_TIMEOUT and stores no output
    spec = spec_for("serving_decode")
    wl, t = _load(spec)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 22).to(DEV)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    ws = _decode_attn_call(spec, t, step, sel)
    torch.cuda.synchronize()
    assert _status(step) == 0
    ws[-8 * spec.n_rows:] = 0x77
    step.out.fill_(3.0)
    _decode_attn_call(spec, t, step, sel, ws)
    torch.cuda.synchronize()
    assert _status(step) & B.CSA_DEV_TIMEOUT
    assert bool((step.out == 3.0).all())
    # zeroed again, the workspace works
    ws[-8 * spec.n_rows:] = 0
    step.status.zero_()
    _decode_attn_call(spec, t, step, sel, ws)
    torch.cuda.synchronize()
    assert _status(step) == 0


@pytest.mark.parametrize("chunk", [[10, 10, 10, 10], [40, 40, 40, 40]])
def test_decode_attention_split_geometries(chunk):
    # 40 rows: three CTAs per row, two tiles each, merged through the
    # workspace; 160 rows (more rows than SMs): one CTA per row, no merge wait
    spec = spec_for("serving_decode", chunk=chunk, topk=512, seed=57)
    _attn_case(spec, 23, False, rows=range(0, spec.n_rows, 7))
