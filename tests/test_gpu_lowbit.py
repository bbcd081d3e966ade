"""Low-bit cache formats on the GPU against the float64 oracle, through the C ABI.

"DeepSeek V4.1 Flash", production cache ABI: the window KV in MXFP8 (E4M3
with E8M0 scales per 32 channels), the compressed KV in packed E2M1 with E4M3
scales per 16 channels, the index keys in packed E2M1 with E8M0 scales per 32
dims; quantised when the compressor publishes, dequantised when the indexer
and the attention read.  Publication is checked code by code (decisions at a
rounding tie may differ, rarely); reads are checked against the oracle on
the same codes, and against the BF16 path on host-dequantised copies of the
same pools (bit-identical: every dequantised value is a BF16 value).
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import step as OS
from parity import (INT8_FLIP_RATE, LSE_ABS, check_bf16, check_lowbit_tied, check_scores,
                    check_topk, score_tolerance)
from workloads import BLOCK, make_workload, random_selection, spec_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefill_csa_compress_gb300 as csa  # noqa: E402
from prefill_csa_compress_gb300.pipeline import CsaStep  # noqa: E402

DEV = torch.device("cuda:0")
_CACHE = {}


def _load(spec):
    key = repr(spec)
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = make_workload(spec)
    wl = _CACHE[key]
    return wl, wl.to(DEV)


# ------------------------------------------------------------------ publication


@pytest.mark.parametrize("n_rows,ratio,dx,d,out", [
    (12, 4, 512, 512, "fp4_e4m3"),    # short chunk: fused kernel, 16-channel groups per CTA
    (600, 2, 512, 512, "fp4_e4m3"),   # long chunk: gate GEMM + pooling kernel
    (12, 4, 128, 128, "fp4_e8m0"),    # fused whole-row kernel, rotated index keys
    (600, 4, 256, 128, "fp4_e8m0"),   # long chunk, rotated
    (12, 2, 256, 512, "fp4_e8m0"),    # 32-channel groups of a 512-channel row: row kernels
    (9, 1, 128, 128, "fp4_e4m3"),
    (12, 4, 128, 128, "mxfp8"),       # FP8 index keys, fused kernel
    (600, 4, 256, 128, "mxfp8"),      # FP8 index keys, long chunk
])
def test_fp4_publication(n_rows, ratio, dx, d, out):
    rng = np.random.default_rng(n_rows * 11 + ratio + d)
    pos0 = 4 * 29 + 1
    positions = np.arange(pos0, pos0 + n_rows, dtype=np.int32)
    row_req = np.zeros(n_rows, np.int32)
    x = torch.from_numpy(rng.standard_normal((n_rows, dx)).astype(np.float32)).bfloat16()
    kv = torch.from_numpy((rng.standard_normal((n_rows, d)) *
                           np.exp(rng.uniform(-3, 3, (1, d)))).astype(np.float32)).bfloat16()
    w = torch.from_numpy((rng.standard_normal((dx, d)) / np.sqrt(dx)).astype(np.float32)).bfloat16()
    ape = torch.from_numpy(rng.standard_normal((ratio, d)).astype(np.float32))
    from workloads import rope_tables
    cos, sin = rope_tables(4096)
    rotate = out in ("fp4_e8m0", "mxfp8")
    group = 16 if out == "fp4_e4m3" else 32
    table = torch.tensor([[2, 0, 3, 1]], dtype=torch.int32)
    codes = torch.zeros((4, BLOCK, d if out == "mxfp8" else d // 2), dtype=torch.uint8,
                        device=DEV)
    scales = torch.zeros((4, BLOCK, d // group), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.csa_compress(x=x.to(DEV), kv=kv.to(DEV), w_gate=w.to(DEV), ape=ape.to(DEV), ratio=ratio,
                     positions=torch.from_numpy(positions).to(DEV),
                     row_req=torch.from_numpy(row_req).to(DEV), block_table=table.to(DEV),
                     out=out, cmp_pool=codes, scale_pool=scales, rotate=rotate,
                     rope_cos=cos.to(DEV), rope_sin=sin.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    trace = []
    ref = O.compress(x, kv, w, ape, ratio, positions, row_req, rotate=rotate, rope_cos=cos,
                     rope_sin=sin, out=out, trace=trace)
    assert len(ref) > 0
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    n_sc = n_code = 0
    fmt = {"mxfp8": "mxfp8", "fp4_e8m0": "e8m0", "fp4_e4m3": "e4m3"}[out]
    for (_, g, rc, rs), rec in zip(ref, trace):
        pg, row = int(table[0, g // BLOCK]), g % BLOCK
        a, b = check_lowbit_tied(gc[pg, row], gs[pg, row], rc, rs, rec, dx, group, fmt)
        n_sc += a
        n_code += b
    assert n_sc <= INT8_FLIP_RATE * len(ref) * d // group + 1, n_sc
    assert n_code <= INT8_FLIP_RATE * len(ref) * d + 2, n_code
    # rows outside the published groups stay zero
    written = {int(table[0, g // BLOCK]) * BLOCK + g % BLOCK for _, g, _, _ in ref}
    flat = gc.reshape(-1, gc.shape[-1])
    others = [i for i in range(flat.shape[0]) if i not in written]
    assert not flat[others].any()


# ------------------------------------------------------------------ indexer


def _check_fp4_index_rows(wl, t, spec, step, rows, sc):
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    pools = {"idx_pool": wl.idx_pool, "idx_kscale": wl.idx_kscale, "cmp_pool": wl.cmp_pool,
             "cmp_scale": wl.cmp_scale}
    sel = step.topk_idx.cpu().numpy()
    kpool = O.LowBitPool(wl.idx_pool, wl.idx_kscale,
                         "mxfp8" if spec.key_fmt == "mxfp8" else "fp4_e8m0")
    for row in rows:
        b = int(wl.row_req[row])
        ref = OS.index_row(wl.t, spec, pools, row)
        V = len(ref)
        keys = O.cache_rows(kpool, wl.cmp_table[b].numpy(), range(V))
        q_rot = O.rope_rotate(wl.q_idx[row], int(wl.row_pos[row]), wl.rope_cos, wl.rope_sin)
        floor = score_tolerance(q_rot, O.as_f64(wl.idx_w[row]), keys, np.ones(V))
        tol = check_scores(sc[row, :V], ref, floor)
        order = np.lexsort((np.arange(V), -sc[row, :V].astype(np.float64)))
        mine = np.sort(order[:spec.topk])
        assert np.array_equal(sel[row][:len(mine)], mine)
        check_topk(sel[row], ref, tol, spec.topk)


@pytest.mark.parametrize("name,over", [
    ("lowbit_decode", {}),
    ("lowbit_decode", dict(ctx=[40000, 3000], chunk=[2, 2], ratio=4, topk=700, seed=91,
                           kv_pool_pages=None, cmp_pool_pages=None)),
    ("lowbit_decode", dict(key_fmt="mxfp8", seed=97)),            # FP8 index keys
    ("lowbit_decode", dict(ctx=[3000], chunk=[80], ratio=4, topk=128, seed=98,
                           kv_pool_pages=None, cmp_pool_pages=None,
                           key_fmt="mxfp8")),                     # FP8, four-row groups
])
def test_fp4_index_parity(name, over):
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    _check_fp4_index_rows(wl, t, spec, step, range(spec.n_rows), scores.cpu().numpy())


def test_fp4_index_prefill_kernel():
    """More than 64 rows: the four-row-group kernel with A tiles in shared memory."""
    spec = spec_for("lowbit_decode", ctx=[3000], chunk=[80], ratio=4, topk=128, seed=92,
                    kv_pool_pages=None, cmp_pool_pages=None)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    _check_fp4_index_rows(wl, t, spec, step, [0, 1, 40, 79], scores.cpu().numpy())


def test_fp4_index_full_size_sampled():
    spec = spec_for("lowbit_million")
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, compress=False)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.empty((spec.n_rows, n_cap), device=DEV)
    step.index(scores=scores)
    _check_fp4_index_rows(wl, t, spec, step, range(spec.n_rows), scores.cpu().numpy())


# ------------------------------------------------------------------ attention


def _dequant_pool_bf16(codes, scales, fmt):
    pool = O.LowBitPool(codes.cpu(), scales.cpu(), fmt)
    P, R = codes.shape[:2]
    vals = pool.dequant_rows(pool.codes.reshape(P * R, -1).numpy(),
                             pool.scales.reshape(P * R, -1).numpy())
    assert np.array_equal(O.bf16_round(vals), vals)  # exactly BF16 values
    return torch.from_numpy(vals.reshape(P, R, -1)).to(torch.bfloat16).to(codes.device)


@pytest.mark.parametrize("name,over,combo", [
    ("lowbit_decode", {}, "both"),
    ("lowbit_decode", {}, "kv"),
    ("lowbit_decode", {}, "cmp"),
    ("lowbit_decode", dict(ctx=[130, 5, 129, 3000], chunk=[3, 5, 2, 7], topk=100, seed=93,
                           pad_rows=2), "both"),
])
def test_lowbit_attention(name, over, combo):
    """Decode attention over low-bit pools: against the oracle on the same
    codes, and bit-identical to the BF16 path on dequantised copies."""
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              if int(wl.row_req[i]) >= 0 else 0 for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 17).to(DEV)
    kv_bf = _dequant_pool_bf16(t["kv_pool"], t["kv_scale"], "mxfp8")
    cmp_bf = _dequant_pool_bf16(t["cmp_pool"], t["cmp_scale"], "fp4_e4m3")
    use_kv_lb, use_cmp_lb = combo in ("both", "kv"), combo in ("both", "cmp")
    outs = []
    for lowbit in (True, False):
        out = torch.zeros_like(t["q"])
        lse = torch.zeros(t["q"].shape[:2], dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        kv_lb, cmp_lb = lowbit and use_kv_lb, lowbit and use_cmp_lb
        csa.csa_sparse_attn_decode(
            q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=sel,
            kv_pool=t["kv_pool"] if kv_lb else kv_bf, kv_block_table=t["kv_table"],
            kv_len=t["kv_len"], cmp_pool=t["cmp_pool"] if cmp_lb else cmp_bf,
            cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"], ratio=spec.ratio, out=out,
            lse=lse, sink=t["sink"], rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
            status=status, kv_scale_pool=t["kv_scale"] if kv_lb else None,
            cmp_scale_pool=t["cmp_scale"] if cmp_lb else None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((out.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    out = outs[0][0].double().numpy()
    lse = outs[0][1].numpy()
    pools = {"cmp_pool": wl.cmp_pool, "cmp_scale": wl.cmp_scale, "idx_pool": wl.idx_pool,
             "idx_kscale": wl.idx_kscale}
    g, r, gl, rl = [], [], [], []
    for row in range(spec.n_rows):
        if int(wl.row_req[row]) < 0:
            continue
        o_ref, l_ref = OS.attention_row(wl.t, spec, pools, row, sel[row].cpu().numpy())
        g.append(out[row])
        r.append(o_ref)
        gl.append(lse[row])
        rl.append(l_ref)
    mag = max(1.0, float(np.max(np.abs(np.stack(r)))) / 2)
    check_bf16(np.stack(g), np.stack(r), "attention out", magnitude=mag)
    assert np.max(np.abs(np.stack(gl) - np.stack(rl))) <= LSE_ABS * max(1.0, np.max(np.abs(rl)))


@pytest.mark.parametrize("over", [
    dict(ctx=[700], chunk=[300], ratio=4, topk=48, seed=94, kv_pool_pages=None,
         cmp_pool_pages=None),
    dict(ctx=[2500, 900], chunk=[130, 70], ratio=2, topk=200, seed=95),
])
def test_lowbit_prefill_attention(over):
    """The prefill call dequantises the low-bit pools into its BF16 arena:
    bit-identical to the BF16 path on dequantised copies, and the oracle's."""
    spec = spec_for("lowbit_decode", **over)
    wl, t = _load(spec)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              if int(wl.row_req[i]) >= 0 else 0 for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 19).to(DEV)
    kv_bf = _dequant_pool_bf16(t["kv_pool"], t["kv_scale"], "mxfp8")
    cmp_bf = _dequant_pool_bf16(t["cmp_pool"], t["cmp_scale"], "fp4_e4m3")
    outs = []
    for lowbit in (True, False):
        out = torch.zeros_like(t["q"])
        lse = torch.zeros(t["q"].shape[:2], dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        csa.csa_sparse_attn_prefill(
            q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=sel,
            kv_pool=t["kv_pool"] if lowbit else kv_bf, kv_block_table=t["kv_table"],
            kv_len=t["kv_len"], cmp_pool=t["cmp_pool"] if lowbit else cmp_bf,
            cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"], ratio=spec.ratio, out=out,
            lse=lse, sink=t["sink"], rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
            status=status, kv_scale_pool=t["kv_scale"] if lowbit else None,
            cmp_scale_pool=t["cmp_scale"] if lowbit else None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((out.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    out = outs[0][0].double().numpy()
    pools = {"cmp_pool": wl.cmp_pool, "cmp_scale": wl.cmp_scale, "idx_pool": wl.idx_pool,
             "idx_kscale": wl.idx_kscale}
    rows = [r for r in range(spec.n_rows) if int(wl.row_req[r]) >= 0][::17]
    g = np.stack([out[r] for r in rows])
    ref = np.stack([OS.attention_row(wl.t, spec, pools, r, sel[r].cpu().numpy())[0]
                    for r in rows])
    check_bf16(g, ref, "prefill out", magnitude=max(1.0, float(np.max(np.abs(ref))) / 2))


# ------------------------------------------------------------------ the step


@pytest.mark.parametrize("name,over", [
    ("lowbit_decode", {}),
    ("lowbit_million", {}),
    ("lowbit_prefill", dict(ctx=[1500], chunk=[1500], seed=96)),   # FP4 publication of 375 groups
    ("lowbit_decode", dict(key_fmt="mxfp8", seed=99)),               # FP8 index keys
    ("lowbit_prefill", dict(ctx=[1500], chunk=[1500], seed=100, overlap=True)),
])
def test_lowbit_step_chain(name, over):
    """compress (FP4 publication) -> FP4 indexer -> low-bit attention, against
    the oracle's chain on the same inputs."""
    spec = spec_for(name, **over)
    wl, t = _load(spec)
    step = CsaStep(t, spec.ratio, spec.topk, prefill=spec.mode == "prefill", overlap=spec.overlap)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rows = list(range(spec.n_rows)) if spec.n_rows <= 8 else [0, 5, 127, 128, 700,
                                                              spec.n_rows - 1]
    trace = {}
    pools, res = OS.full_step(wl.t, spec, rows=rows, trace=trace)
    # the published entries: codes like the oracle's except at rounding ties
    table = wl.cmp_table.numpy()
    kfmt = "mxfp8" if spec.key_fmt == "mxfp8" else "e8m0"
    for name, scale_name, out_key, tr_key, d, group, fmt in (
            ("cmp_pool", "cmp_scale", "main_out", "main", spec.head_dim, 16, "e4m3"),
            ("idx_pool", "idx_kscale", "idx_out", "idx", spec.idx_dim, 32, kfmt)):
        gc, gs = t[name].cpu().numpy(), t[scale_name].cpu().numpy()
        n_code = 0
        for (b, g, rc, rs), rec in zip(trace[out_key], trace[tr_key]):
            pg = int(table[b, g // BLOCK])
            n_code += check_lowbit_tied(gc[pg, g % BLOCK], gs[pg, g % BLOCK], rc, rs, rec, d,
                                        group, fmt)[1]
        assert n_code <= INT8_FLIP_RATE * max(1, len(trace[out_key])) * d + 2, (name, n_code)
    kpool_ref = O.LowBitPool(pools["idx_pool"], pools["idx_kscale"],
                             "mxfp8" if spec.key_fmt == "mxfp8" else "fp4_e8m0")
    kpool_gpu = O.LowBitPool(t["idx_pool"].cpu(), t["idx_kscale"].cpu(),
                             "mxfp8" if spec.key_fmt == "mxfp8" else "fp4_e8m0")
    sel = step.topk_idx.cpu().numpy()
    out = step.out.cpu().double().numpy()
    g_out, r_out = [], []
    for row, rr in res.items():
        s_ref = rr["scores"]
        V = len(s_ref)
        if V == 0:  # no compressed entry visible yet
            assert np.all(sel[row] == -1)
        else:
            # 1e-4 relative or the cancellation floor, plus the exact score
            # change of keys the two sides published differently
            b = int(wl.row_req[row])
            q_rot = O.rope_rotate(wl.q_idx[row], int(wl.row_pos[row]), wl.rope_cos, wl.rope_sin)
            w = O.as_f64(wl.idx_w[row])
            keys = O.cache_rows(kpool_ref, table[b], range(V))
            tol = np.maximum(1e-4 * np.abs(s_ref),
                             score_tolerance(q_rot, w, keys, np.ones(V)))
            dk = np.abs(O.cache_rows(kpool_gpu, table[b], range(V)) - keys)
            moved = np.nonzero(dk.any(axis=1))[0]
            if len(moved):
                tol[moved] += (dk[moved] @ np.abs(q_rot).T) @ np.abs(w) * 1.001
            check_topk(sel[row], s_ref, tol, spec.topk)
        # attention on the GPU's accepted selection, every checked row
        g_out.append(out[row])
        r_out.append(OS.attention_row(wl.t, spec, pools, row, sel[row])[0])
    check_bf16(np.stack(g_out), np.stack(r_out), "out",
               magnitude=max(1.0, float(np.max(np.abs(np.stack(r_out)))) / 2))
