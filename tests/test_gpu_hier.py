"""Hierarchical indexer on the GPU against the float64 oracle, through the C ABI.

Level one ("DeepSeek V4.1 Flash", hierarchical indexer): besides its top-k,
the indexer selects the candidate blocks with the largest block maxima.
Reindex: a later layer scores only the positions of those blocks and selects
its top-k among them.  As for the flat indexer, a selection is checked twice:
exactly against the oracle's selection rule applied to the scores the kernel
computed (the integer decision taken in the kernel's precision), and as a
valid selection under the oracle's float64 scores within the score tolerance.
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import step as OS
from parity import LSE_ABS, check_bf16, check_scores, check_topk, score_tolerance
from workloads import BLOCK, make_workload, reindex_view, spec_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from prefill_csa_compress_gb300.pipeline import CsaStep, StepChain  # noqa: E402

DEV = torch.device("cuda:0")
BAD_INDEX = 0x4

_CACHE = {}


def _load(spec):
    key = repr(spec)
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = make_workload(spec)
    wl = _CACHE[key]
    return wl, wl.to(DEV)


def _pools(wl):
    p = {"cmp_pool": wl.cmp_pool, "idx_pool": wl.idx_pool, "idx_scale": wl.idx_scale}
    if "idx_kscale" in wl.t:
        p.update(idx_kscale=wl.idx_kscale, cmp_scale=wl.cmp_scale)
    return p


def _floor(t, row, pools, positions):
    """Score tolerance floor of ``positions`` of row ``row`` (layer tensors ``t``)."""
    b = int(t["row_req"][row])
    p = int(t["row_pos"][row])
    table = t["cmp_table"][b].numpy()
    if "idx_kscale" in pools:  # FP4 keys: dequantised, unit scale
        keys = O.cache_rows(O.LowBitPool(pools["idx_pool"], pools["idx_kscale"], "fp4_e8m0"),
                            table, positions)
        scl = np.ones(len(keys))
    else:
        keys = O.page_rows(pools["idx_pool"], table, positions)
        scl = O.page_rows(pools["idx_scale"], table, positions)
    q_rot = O.rope_rotate(t["q_idx"][row], p, t["rope_cos"], t["rope_sin"])
    return score_tolerance(q_rot, O.as_f64(t["idx_w"][row]), keys, scl)


def _valid_prefix(c, nb):
    n = 0
    while n < len(c) and 0 <= c[n] < nb and (n == 0 or c[n] > c[n - 1]):
        n += 1
    return n


def _level_one(spec, t):
    step = CsaStep(t, spec.ratio, spec.topk, compress=False, n_cand=spec.n_cand,
                   cand_block=spec.cand_block)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return step, scores.cpu().numpy()


def _check_level_one(wl, spec, step, sc, rows):
    cb = spec.cand_block
    cand = step.cand.cpu().numpy()
    for row in rows:
        if int(wl.row_req[row]) < 0:
            assert np.all(cand[row] == -1)
            continue
        ref = OS.index_row(wl.t, spec, _pools(wl), row)
        V = len(ref)
        tol = check_scores(sc[row, :V], ref, _floor(wl.t, row, _pools(wl), range(V)))
        # exactly the level-one rule applied to the kernel's own scores
        mine = O.select_blocks(sc[row, :V].astype(np.float64), spec.n_cand, cb)
        assert np.array_equal(cand[row], mine), row
        # a valid block selection under the oracle's scores: a block maximum
        # moves by at most the largest tolerance inside the block
        nb = (V + cb - 1) // cb
        bmax = np.array([ref[i * cb:(i + 1) * cb].max() for i in range(nb)])
        btol = np.array([tol[i * cb:(i + 1) * cb].max() for i in range(nb)])
        check_topk(cand[row], bmax, btol, spec.n_cand)


def _reindex(spec, t, cand):
    step = CsaStep(reindex_view(t), spec.ratio, spec.topk, compress=False, cand_in=cand,
                   cand_block=spec.cand_block)
    scores = torch.full((spec.n_rows, cand.shape[1] * spec.cand_block), float("nan"),
                        device=DEV)
    step.index(scores=scores)
    torch.cuda.synchronize()
    return step, scores.cpu().numpy()


def _check_reindex(wl, spec, step, sc, cand, rows):
    cb, k = spec.cand_block, spec.topk
    t2 = OS.reindex_tensors(wl.t)
    sel = step.topk_idx.cpu().numpy()
    ts = step.topk_score.cpu().numpy()
    for row in rows:
        if int(wl.row_req[row]) < 0:
            assert np.all(sel[row] == -1)
            continue
        ref = OS.index_row(t2, spec, _pools(wl), row)
        V = len(ref)
        nv = _valid_prefix(cand[row], (V + cb - 1) // cb)
        pos = np.array([blk * cb + i for blk in cand[row][:nv] for i in range(cb)
                        if blk * cb + i < V], dtype=np.int64)
        if len(pos) == 0:
            assert np.all(sel[row] == -1)
            continue
        got = sc[row, :len(pos)].astype(np.float64)
        tol = check_scores(got, ref[pos], _floor(t2, row, _pools(wl), pos))
        # exactly the reindex rule applied to the kernel's own scores
        full = np.full(V, np.nan)
        full[pos] = got
        mine = O.topk_in_blocks(full, cand[row][:nv], k, cb)
        assert np.array_equal(sel[row], mine), row
        chosen = sel[row][sel[row] >= 0]
        assert np.array_equal(ts[row][:len(chosen)], full[chosen].astype(np.float32))
        # a valid selection under the oracle's scores, in candidate order
        where = {int(p): i for i, p in enumerate(pos)}
        comp = np.array([where[int(p)] if p >= 0 else -1 for p in sel[row]])
        check_topk(comp, ref[pos], tol, k)


HIER_SMALL = [
    # long main top-k rows (n_cap 10112), short block rows; a 3-row request
    dict(ctx=[40000, 30001, 9000, 700], chunk=[2, 2, 1, 3], n_cand=256, seed=71),
    # 16-position blocks; more candidate blocks than some rows have
    dict(ctx=[12000, 2500], chunk=[2, 2], n_cand=300, cand_block=16, topk=256, seed=72),
    # 32-position blocks, padding rows, every block a candidate for short rows
    dict(ctx=[5000, 100], chunk=[2, 1], n_cand=64, cand_block=32, topk=128, seed=73,
         pad_rows=2),
    # FP4 index keys (low-bit caches): the gathered copies of 64-byte key rows
    dict(ctx=[40000, 9000], chunk=[2, 2], n_cand=200, topk=256, seed=78, lowbit=True),
]


@pytest.mark.parametrize("over", HIER_SMALL)
def test_level_one_parity(over):
    spec = spec_for("hier_decode", **over)
    wl, t = _load(spec)
    step, sc = _level_one(spec, t)
    _check_level_one(wl, spec, step, sc, range(spec.n_rows))


@pytest.mark.parametrize("over", HIER_SMALL)
def test_reindex_parity(over):
    """Reindex inside the GPU's own level-one candidates."""
    spec = spec_for("hier_decode", **over)
    wl, t = _load(spec)
    step1, _ = _level_one(spec, t)
    step2, sc2 = _reindex(spec, t, step1.cand)
    assert int(step2.status.item()) == 0
    _check_reindex(wl, spec, step2, sc2, step1.cand.cpu().numpy(), range(spec.n_rows))


def test_reindex_given_candidates():
    """Seeded candidate lists (an input): sparse blocks spread over the whole
    context, shorter lists padded with -1, and the ragged last block."""
    spec = spec_for("hier_decode", ctx=[20000, 9001], chunk=[2, 2], n_cand=96, topk=200,
                    seed=74)
    wl, t = _load(spec)
    rng = np.random.default_rng(75)
    cand = np.full((spec.n_rows, spec.n_cand), -1, dtype=np.int32)
    for row in range(spec.n_rows):
        b, p = int(wl.row_req[row]), int(wl.row_pos[row])
        V = O.visible_count(p, spec.ratio, int(wl.n_cmp[b]))
        nb = (V + 7) // 8
        m = [spec.n_cand, 40, spec.n_cand, 1][row]
        blocks = np.sort(rng.choice(nb - 1, size=m - 1, replace=False))
        cand[row, :m] = np.append(blocks, nb - 1)  # the last, ragged block is always in
    cand_d = torch.from_numpy(cand).to(DEV)
    step2, sc2 = _reindex(spec, t, cand_d)
    assert int(step2.status.item()) == 0
    _check_reindex(wl, spec, step2, sc2, cand, range(spec.n_rows))


def test_reindex_malformed_candidates_flag_and_truncate():
    """A list is used up to its first entry that is not a strictly ascending
    visible block; a later entry other than -1 raises CSA_DEV_BAD_INDEX."""
    spec = spec_for("hier_decode", ctx=[20000, 16000], chunk=[2, 2], n_cand=8, topk=24,
                    seed=76)
    wl, t = _load(spec)
    cand = np.array([
        [5, 9, 3, 40, -1, -1, -1, -1],         # descends at entry 2
        [-1, 4, 6, -1, -1, -1, -1, -1],        # nothing before the -1
        [2, 7, 10 ** 6, 11, -1, -1, -1, -1],   # a block past the visible ones
        [1, 2, 3, 4, 5, 6, 7, 8],              # valid
    ], dtype=np.int32)
    step2, sc2 = _reindex(spec, t, torch.from_numpy(cand).to(DEV))
    assert int(step2.status.item()) & BAD_INDEX
    _check_reindex(wl, spec, step2, sc2, cand, range(spec.n_rows))


def test_hier_full_size_sampled():
    """1,048,576 positions: 262,144 entries per row (multi-CTA top-k), 32,768
    blocks (multi-CTA block top-k), 16,384 candidate entries per reindex row."""
    spec = spec_for("hier_decode")
    wl, t = _load(spec)
    step1, sc = _level_one(spec, t)
    _check_level_one(wl, spec, step1, sc, [0, 5])
    step2, sc2 = _reindex(spec, t, step1.cand)
    assert int(step2.status.item()) == 0
    _check_reindex(wl, spec, step2, sc2, step1.cand.cpu().numpy(), [0, 5, 7])


@pytest.mark.parametrize("over", [
    dict(ctx=[40000, 30001], chunk=[2, 2], n_cand=256, seed=77),
    {},
])
def test_hier_layer_chain(over):
    """Level-one layer (compressors, indexer with candidate blocks,
    attention) then reindex layer (indexer inside the candidates, attention)
    as one step, against the oracle's chain."""
    spec = spec_for("hier_decode", **over)
    wl, t = _load(spec)
    s1 = CsaStep(t, spec.ratio, spec.topk, n_cand=spec.n_cand, cand_block=spec.cand_block)
    s2 = CsaStep(reindex_view(t), spec.ratio, spec.topk, compress=False, cand_in=s1.cand,
                 cand_block=spec.cand_block, status_buf=s1.status)
    chain = StepChain([s1, s2]).prepare()
    chain.run()
    torch.cuda.synchronize()
    assert int(chain.status.item()) == 0
    rows = [0, 3] if spec.n_rows > 4 else list(range(spec.n_rows))
    _, res = OS.full_step(wl.t, spec, rows=rows)
    sel1, sel2 = s1.topk_idx.cpu().numpy(), s2.topk_idx.cpu().numpy()
    out1, out2 = s1.out.cpu().double().numpy(), s2.out.cpu().double().numpy()
    lse2 = s2.lse.cpu().numpy()
    same = 0
    for row, rr in res.items():
        # selections: valid under the oracle's scores (loose: the pools the
        # compressor wrote may differ from the oracle's by a rounded code)
        s_ref = rr["scores"]
        tol = np.maximum(1e-3 * np.abs(s_ref), 1e-3 * np.max(np.abs(s_ref)))
        check_topk(sel1[row], s_ref, tol, spec.topk)
        if np.array_equal(sel1[row], rr["topk"]):
            check_bf16(out1[row], rr["out"], f"row {row} level-one out")
        if np.array_equal(s1.cand[row].cpu().numpy(), rr["cand"]) and \
                np.array_equal(sel2[row], rr["topk2"]):
            same += 1
            check_bf16(out2[row], rr["out2"], f"row {row} reindex out")
            assert np.max(np.abs(lse2[row] - rr["lse2"])) <= LSE_ABS * max(
                1.0, np.max(np.abs(rr["lse2"])))
    assert same >= 1
