"""Data errors on the GPU: each kernel skips the offending element, raises its
bit in the caller's status word and leaves everything else as the oracle has
it (include/csa.h: CSA_DEV_BAD_BLOCK, CSA_DEV_BAD_POS, CSA_DEV_BAD_INDEX,
CSA_DEV_POS_GE_CAP).  Every bad value here is one the kernels check before
any access, so nothing is read or written out of bounds.
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import step as OS
from parity import check_bf16, check_scores, score_tolerance
from workloads import BLOCK, make_workload, random_selection, spec_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefill_csa_compress_gb300 as csa  # noqa: E402
from prefill_csa_compress_gb300.pipeline import CsaStep  # noqa: E402

DEV = torch.device("cuda:0")
BAD_BLOCK, BAD_POS, BAD_INDEX, POS_GE_CAP = 0x1, 0x2, 0x4, 0x8


def _spec():
    return spec_for("serving_decode", topk=64, seed=81)


def test_attention_flags_bad_entries_and_skips_them():
    spec = _spec()
    wl = make_workload(spec)
    t = wl.to(DEV)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 3)
    sel[0, 5] = limits[0] + 7           # past the row's visible entries
    sel[1, 0] = -1                      # an ordinary hole
    t_bad = dict(t)
    kv_len = wl.kv_len.clone()
    kv_len[1] = int(wl.row_pos[2]) - 3  # request 1's window runs past its length
    t_bad["kv_len"] = kv_len.to(DEV)
    step = CsaStep(t_bad, spec.ratio, spec.topk, compress=False)
    step.attention(topk_idx=sel.to(DEV))
    torch.cuda.synchronize()
    st = int(step.status.item())
    assert st & BAD_INDEX and st & BAD_POS and not st & BAD_BLOCK
    out = step.out.cpu().double().numpy()
    assert np.all(np.isfinite(out))
    # row 0 equals the oracle over its valid entries; the rows of request 1
    # equal the oracle over window positions below the shortened length
    pools = {"cmp_pool": wl.cmp_pool}
    sel0 = sel[0].numpy().copy()
    sel0[sel0 >= limits[0]] = -1
    o_ref, _ = OS.attention_row(wl.t, spec, pools, 0, sel0)
    check_bf16(out[0], o_ref, "row 0")
    b = int(wl.row_req[2])
    for row in (2, 3):
        p = int(wl.row_pos[row])
        s_ = sel[row].numpy()
        ks = [O.page_rows(wl.cmp_pool, wl.cmp_table[b].numpy(), [c])[0] for c in s_ if c >= 0]
        ws = [O.page_rows(wl.kv_pool, wl.kv_table[b].numpy(), [q])[0]
              for q in O.window_positions(p) if q < int(kv_len[b])]
        K = np.stack(ks + ws)
        q_rot = O.rope_rotate(wl.q[row], p, wl.rope_cos, wl.rope_sin)
        logit = (q_rot @ K.T) / np.sqrt(512)
        m = np.maximum(logit.max(axis=1), O.as_f64(wl.sink))
        e = np.exp(logit - m[:, None])
        den = e.sum(axis=1) + np.exp(O.as_f64(wl.sink) - m)
        check_bf16(out[row], (e @ K) / den[:, None], f"row {row}")


def test_attention_flags_unmapped_pages():
    spec = _spec()
    wl = make_workload(spec)
    t = wl.to(DEV)
    limits = [O.visible_count(int(wl.row_pos[i]), spec.ratio, int(wl.n_cmp[int(wl.row_req[i])]))
              for i in range(spec.n_rows)]
    sel = random_selection(limits, spec.topk, 4)
    table = wl.cmp_table.clone()
    table[0, 0] = int(wl.cmp_pool.shape[0]) + 5  # beyond the pool: flagged, never read
    t_bad = dict(t)
    t_bad["cmp_table"] = table.to(DEV)
    step = CsaStep(t_bad, spec.ratio, spec.topk, compress=False)
    step.attention(topk_idx=sel.to(DEV))
    torch.cuda.synchronize()
    assert int(step.status.item()) & BAD_BLOCK
    assert np.all(np.isfinite(step.out.cpu().double().numpy()))


def test_indexer_flags_unmapped_pages_and_scores_the_rest():
    spec = _spec()
    wl = make_workload(spec)
    t = wl.to(DEV)
    table = wl.cmp_table.clone()
    table[0, 1] = -1                      # request 0's second page
    t_bad = dict(t)
    t_bad["cmp_table"] = table.to(DEV)
    step = CsaStep(t_bad, spec.ratio, spec.topk, compress=False)
    n_cap = table.shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    step.index(scores=scores)
    torch.cuda.synchronize()
    assert int(step.status.item()) & BAD_BLOCK
    sc = scores.cpu().numpy()
    pools = {"idx_pool": wl.idx_pool, "idx_scale": wl.idx_scale, "cmp_pool": wl.cmp_pool}
    ref = OS.index_row(wl.t, spec, pools, 0)
    V = len(ref)
    # the unmapped page's entries score -inf (never selected); the others as the oracle
    assert np.all(sc[0, BLOCK:2 * BLOCK] == -np.inf)
    keep = np.r_[0:BLOCK, 2 * BLOCK:V]
    keys = O.page_rows(wl.idx_pool, wl.cmp_table[0].numpy(), keep)
    scl = O.page_rows(wl.idx_scale, wl.cmp_table[0].numpy(), keep)
    q_rot = O.rope_rotate(wl.q_idx[0], int(wl.row_pos[0]), wl.rope_cos, wl.rope_sin)
    check_scores(sc[0, keep], ref[keep], score_tolerance(q_rot, O.as_f64(wl.idx_w[0]), keys, scl))
    sel = step.topk_idx.cpu().numpy()[0]
    assert not np.any((sel >= BLOCK) & (sel < 2 * BLOCK))


def test_positions_beyond_the_rope_table_are_flagged():
    spec = _spec()
    wl = make_workload(spec)
    t = wl.to(DEV)
    cap = int(wl.row_pos[0])  # rows of request 0 (and later positions) fall outside
    t_bad = dict(t)
    t_bad["rope_cos"] = t["rope_cos"][:cap].contiguous()
    t_bad["rope_sin"] = t["rope_sin"][:cap].contiguous()
    step = CsaStep(t_bad, spec.ratio, spec.topk, compress=False)
    step.index()
    step.attention()
    torch.cuda.synchronize()
    assert int(step.status.item()) & POS_GE_CAP
    assert np.all(np.isfinite(step.out.cpu().double().numpy()))


def test_compressor_flags_unmapped_destination_and_writes_nothing_there():
    spec = spec_for("chunked_prefill", ctx=[300], chunk=[300], seed=82)
    wl = make_workload(spec)
    t = wl.to(DEV)
    table = wl.cmp_table.clone()
    table[0, 0] = -1  # every group of the chunk lands in page 0
    t_bad = dict(t)
    t_bad["cmp_table"] = table.to(DEV)
    before = t["cmp_pool"].clone()
    step = CsaStep(t_bad, spec.ratio, spec.topk, prefill=True)
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) & BAD_BLOCK
    assert torch.equal(t["cmp_pool"], before)


def test_empty_batches_launch_nothing():
    spec = _spec()
    wl = make_workload(spec)
    t = wl.to(DEV)
    empty = {k: (v[:0] if k in ("q", "q_idx", "idx_w", "kv_raw", "idx_raw", "row_req", "row_pos")
                 else v) for k, v in t.items()}
    step = CsaStep(empty, spec.ratio, spec.topk)
    n0 = csa.launch_count()
    step.run()
    torch.cuda.synchronize()
    assert csa.launch_count() == n0
    assert int(step.status.item()) == 0


def test_ring_compressor_flags_unmapped_destination_and_still_updates_the_ring():
    """The short-chunk compressor with state rings (overlapping windows): a
    group whose destination page is unmapped is flagged and not written,
    while the rings still receive every row as the oracle's rings do."""
    spec = spec_for("overlap_decode", seed=83)
    wl = make_workload(spec)
    t = wl.to(DEV)
    assert int(wl.row_req[1]) == 0 and int(wl.row_pos[1]) % spec.ratio == spec.ratio - 1
    g0 = int(wl.row_pos[1]) // spec.ratio  # the group row 1 closes
    table = wl.cmp_table.clone()
    table[0, g0 // BLOCK] = -1
    t_bad = dict(t)
    t_bad["cmp_table"] = table.to(DEV)
    before = t["cmp_pool"].clone()
    step = CsaStep(t_bad, spec.ratio, spec.topk, overlap=True)
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) & BAD_BLOCK
    pools, main, _ = OS.compress_step(wl.t, spec)
    got = t["cmp_pool"].cpu()
    ref_table = wl.cmp_table.numpy()
    n_other = 0
    for b, g, y in main:
        pg, row = int(ref_table[b, g // BLOCK]), g % BLOCK
        if b == 0 and g == g0:
            assert torch.equal(got[pg, row], before[pg, row].cpu())
        else:
            check_bf16(got[pg, row].double().numpy(), y, f"entry {b}/{g}")
            n_other += 1
    assert n_other > 0
    for name in ("state_main", "state_idx"):
        got_s = t[name].cpu().double().numpy()
        ref_s = pools[name]
        d = got_s.shape[2] // 2
        assert np.array_equal(got_s[..., :d], ref_s[..., :d]), name
        err = np.abs(got_s[..., d:] - ref_s[..., d:])
        assert np.all(err <= 1e-4 * np.maximum(1.0, np.abs(ref_s[..., d:]))), (name, err.max())


def test_cooperative_topk_wait_gives_up_and_the_next_call_succeeds():
    """The bounded barrier wait of the cooperative top-k (rows longer than
    16384 entries): with wait_limit_ns < 0 every
    CTA that is not the last to reach a barrier gives up at once, raises
    CSA_DEV_TIMEOUT and stops; the call returns, the context stays usable and
    the next call (default limit) selects exactly the (score desc, index asc)
    top-k of its scores."""
    spec = spec_for("ratio1_decode", ctx=[40000, 30000], chunk=[2, 2], topk=512, seed=83)
    wl = make_workload(spec)
    t = wl.to(DEV)
    TIMEOUT = 0x10
    n_cap = t["cmp_table"].shape[1] * BLOCK

    def call(limit):
        idx = torch.full((spec.n_rows, spec.topk), -7, dtype=torch.int32, device=DEV)
        sc = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        csa.csa_index_topk(q_idx=t["q_idx"], weights=t["idx_w"], row_req=t["row_req"],
                           row_pos=t["row_pos"], n_cmp=t["n_cmp"], ratio=spec.ratio,
                           idx_pool=t["idx_pool"], idx_scale_pool=t["idx_scale"],
                           cmp_block_table=t["cmp_table"], topk=spec.topk, topk_idx=idx,
                           scores=sc, rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
                           mode=csa.CSA_MODE_PREFILL, status=st, wait_limit_ns=limit)
        torch.cuda.synchronize()
        return idx.cpu().numpy(), sc.cpu().numpy(), int(st.item())

    _, _, st = call(-1)
    assert st & TIMEOUT
    got, sc, st = call(0)
    assert st == 0
    for row in range(spec.n_rows):
        b = int(wl.row_req[row])
        V = O.visible_count(int(wl.row_pos[row]), spec.ratio, int(wl.n_cmp[b]))
        assert V > 16384
        mine = np.sort(np.lexsort((np.arange(V), -sc[row, :V].astype(np.float64)))[:spec.topk])
        assert np.array_equal(got[row], mine)
