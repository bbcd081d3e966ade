"""The whole step at full size, against the oracle's own chain, for each of
the five configurations.

One ``CsaStep`` (both compressors, the indexer top-k, the sparse attention)
runs on the GPU over the configuration's full workload; the oracle runs its
own chain (``oracle.step.full_step``) over the same inputs.  Checked, for
every decode row and for the prefill chunk's rows at and around tile edges:

* publication: every group the step's compressors publish (BF16 rows within
  the BF16 bounds; INT8 index keys code by code, a differing code only at a
  rounding tie the oracle's trace locates);
* indexer scores: each visible entry within 1e-4 relative (or the
  cancellation floor), plus the exact score change of any key that the two
  sides published differently;
* top-k: exactly the (score desc, index asc) selection of the kernel's own
  scores, and accepted against the oracle's scores ("DeepSeek V4.1 Flash",
  Top-K acceptance: eligibility, uniqueness, ascending positions, trailing
  -1, cutoff quality, and the oracle's set wherever its boundary is clear);
* attention: the output and lse against the oracle recomputed for the
  GPU's own accepted selection, on every checked row.
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import step as OS
from parity import (LSE_ABS, check_bf16, check_int8_tied, check_scores, check_topk,
                    score_tolerance)
from workloads import BLOCK, make_workload, spec_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from prefill_csa_compress_gb300.pipeline import CsaStep  # noqa: E402

DEV = torch.device("cuda:0")

# rows of the 8192-token prefill chunk: both sides of the 128-row tile edges,
# the first rows (no compressed entry visible yet), the 512- and
# 2048-entry marks of the visible count, and the last rows
PREFILL_ROWS = [0, 1, 2, 3, 4, 5, 126, 127, 128, 129, 255, 256, 511, 512, 1023, 1024, 2046,
                2047, 2048, 2049, 4095, 4096, 6143, 6144, 8190, 8191]


def _rows(spec, wl):
    if spec.mode == "prefill":
        return PREFILL_ROWS
    return [r for r in range(spec.n_rows) if int(wl.row_req[r]) >= 0]


def _dequant_keys(pool, scale, table_row, V):
    keys = O.page_rows(pool, table_row, range(V))
    scl = O.page_rows(scale, table_row, range(V))
    return keys, scl


@pytest.mark.parametrize("name", ["tiny_decode", "serving_decode", "ratio1_decode",
                                  "million_decode", "chunked_prefill"])
def test_full_size_step_chain(name):
    spec = spec_for(name)
    wl = make_workload(spec)
    t = wl.to(DEV)
    prefill = spec.mode == "prefill"
    step = CsaStep(t, spec.ratio, spec.topk, prefill=prefill, overlap=spec.overlap)
    n_cap = t["cmp_table"].shape[1] * BLOCK
    scores = torch.full((spec.n_rows, n_cap), float("nan"), device=DEV)
    # the calls of CsaStep.run(), with a caller score buffer for the indexer
    step.compress()
    step.index(scores=scores)
    step.attention()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rows = _rows(spec, wl)
    trace = {}
    pools, res = OS.full_step(wl.t, spec, rows=rows, trace=trace)

    # ---- publication
    table = wl.cmp_table.numpy()
    got_cmp = t["cmp_pool"].cpu()
    got_idx = t["idx_pool"].cpu()
    got_isc = t["idx_scale"].cpu()
    g_rows, r_rows = [], []
    for b, g, vals in trace["main_out"]:
        g_rows.append(got_cmp[int(table[b, g // BLOCK]), g % BLOCK].double().numpy())
        r_rows.append(vals)
    if g_rows:
        check_bf16(np.stack(g_rows), np.stack(r_rows), "published cmp_kv")
    n_flip = 0
    assert len(trace["idx_out"]) == len(trace["idx"])
    for (b, g, codes, scale), rec in zip(trace["idx_out"], trace["idx"]):
        pg = int(table[b, g // BLOCK])
        n_flip += check_int8_tied(got_idx[pg, g % BLOCK].numpy(), got_isc[pg, g % BLOCK].item(),
                                  codes, np.float32(scale), rec, spec.idx_dim)
    n_pub = len(trace["idx_out"])
    if prefill:
        assert n_pub == spec.ctx[0] // spec.ratio

    # ---- per row: scores, selection, attention on the GPU's selection
    sel = step.topk_idx.cpu().numpy()
    sc_all = scores.cpu().numpy()
    out = step.out.cpu().double().numpy()
    lse = step.lse.cpu().numpy()
    g_out, r_out, g_lse, r_lse = [], [], [], []
    for row in rows:
        rr = res[row]
        b = int(wl.row_req[row])
        s_ref = rr["scores"]
        V = len(s_ref)
        q_rot = O.rope_rotate(wl.q_idx[row], int(wl.row_pos[row]), wl.rope_cos, wl.rope_sin)
        w = O.as_f64(wl.idx_w[row])
        keys, scl = _dequant_keys(pools["idx_pool"], pools["idx_scale"], table[b], V)
        tol = np.maximum(1e-4 * np.abs(s_ref), score_tolerance(q_rot, w, keys, scl))
        # keys the two sides published differently move the score by exactly
        # sum_h |w_h| |q_h . dk| at most (ReLU is 1-Lipschitz)
        gk, gs = _dequant_keys(got_idx, got_isc, table[b], V)
        dk = np.abs(gk * gs[:, None] - keys * scl[:, None])
        moved = np.nonzero(dk.any(axis=1))[0]
        if len(moved):
            tol[moved] += (dk[moved] @ np.abs(q_rot).T) @ np.abs(w) * 1.001
        if V:
            check_scores(sc_all[row, :V], s_ref, tol)
            mine = np.sort(np.lexsort((np.arange(V), -sc_all[row, :V].astype(np.float64)))
                           [:spec.topk])
            assert np.array_equal(sel[row][:len(mine)], mine), f"row {row}: not its own top-k"
        check_topk(sel[row], s_ref, tol, spec.topk)
        o_ref, l_ref = OS.attention_row(wl.t, spec, pools, row, sel[row])
        g_out.append(out[row])
        r_out.append(o_ref)
        g_lse.append(lse[row])
        r_lse.append(l_ref)
    check_bf16(np.stack(g_out), np.stack(r_out), "attention out",
               magnitude=max(1.0, float(np.max(np.abs(np.stack(r_out)))) / 2))
    gl, rl = np.stack(g_lse), np.stack(r_lse)
    assert np.max(np.abs(gl - rl)) <= LSE_ABS * max(1.0, float(np.max(np.abs(rl))))
    assert n_flip <= 1e-3 * max(1, n_pub) * spec.idx_dim + 2
