"""Whole-step drivers over a ``workloads.Workload`` — test infrastructure only.

They chain the oracle's definitions in the order the V4 decode layer calls
them ("DeepSeek V4-Flash, MTP point", "Attention paths": main compressor,
index-key compressor, indexer, sparse attention) and never touch the CUDA
library.
"""

from __future__ import annotations

import numpy as np
import torch

from . import csa_oracle as O


def clone_pools(t):
    keys = ("cmp_pool", "idx_pool", "idx_scale", "cmp_scale", "idx_kscale")
    return {k: t[k].clone() for k in keys if k in t}


def _lowbit(t):
    return "cmp_scale" in t


def _key_fmt(t):
    """Low-bit index keys: "fp4_e8m0" (64 bytes a key) or "mxfp8" (128)."""
    return "mxfp8" if t["idx_pool"].shape[-1] == t["q_idx"].shape[-1] else "fp4_e8m0"


def _idx_pool(t, pools):
    """The index-key pool as the oracle reads it (low-bit keys: a LowBitPool)."""
    if _lowbit(t):
        return O.LowBitPool(pools["idx_pool"], pools["idx_kscale"], _key_fmt(t))
    return pools["idx_pool"]


def _kv_pools(t, pools):
    """(window pool, compressed pool) as the oracle reads them."""
    if _lowbit(t):
        return (O.LowBitPool(t["kv_pool"], t["kv_scale"], "mxfp8"),
                O.LowBitPool(pools["cmp_pool"], pools["cmp_scale"], "fp4_e4m3"))
    return t["kv_pool"], pools["cmp_pool"]


def compress_step(t, spec, pools=None, trace=None):
    """Run both compressors over the chunk and publish into (cloned) pools.
    With state rings (``spec.state``) the compressors read and update copies
    of them, returned in pools["state_main"] / pools["state_idx"] (float64).
    ``trace`` (a dict, or None) receives the compressors' trace records
    (``trace["main"]``, ``trace["idx"]``, see ``compress``) and their results
    (``trace["main_out"]``, ``trace["idx_out"]``).

    Returns (pools, main_results, idx_results)."""
    tr_main = tr_idx = None
    if trace is not None:
        tr_main = trace.setdefault("main", [])
        tr_idx = trace.setdefault("idx", [])
    pools = clone_pools(t) if pools is None else pools
    lowbit = _lowbit(t)
    ov = bool(getattr(spec, "overlap", False))
    idx_kw = dict(rotate=True, rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
                  rope_dim=spec.rope_dim, out=_key_fmt(t) if lowbit else "int8", overlap=ov)
    main_out = "fp4_e4m3" if lowbit else "bf16"
    if spec.state:
        pools["state_main"] = O.as_f64(t["state_main"]).copy()
        table = t["state_table"].numpy()
        main = O.compress_stateful(t["kv_raw"], t["kv_raw"], t["w_gate"], t["ape"], spec.ratio,
                                   t["row_pos"], t["row_req"], pools["state_main"], table,
                                   out=main_out, overlap=ov, trace=tr_main)
        idx = []
        if not spec.dense:  # HCA has no indexer, hence no index-key compressor
            pools["state_idx"] = O.as_f64(t["state_idx"]).copy()
            idx = O.compress_stateful(t["idx_raw"], t["idx_raw"], t["w_gate_i"], t["ape_i"],
                                      spec.ratio, t["row_pos"], t["row_req"], pools["state_idx"],
                                      table, trace=tr_idx, **idx_kw)
    else:
        main = O.compress(t["kv_raw"], t["kv_raw"], t["w_gate"], t["ape"], spec.ratio,
                          t["row_pos"], t["row_req"], out=main_out, overlap=ov, trace=tr_main)
        idx = [] if spec.dense else O.compress(t["idx_raw"], t["idx_raw"], t["w_gate_i"],
                                                 t["ape_i"], spec.ratio, t["row_pos"],
                                                 t["row_req"], trace=tr_idx, **idx_kw)
    if trace is not None:
        trace["main_out"], trace["idx_out"] = main, idx
    table = t["cmp_table"].numpy()
    if lowbit:  # packed codes and scale bytes
        for b, g, codes, sb in main:
            pg = int(table[b, g // O.BLOCK])
            pools["cmp_pool"][pg, g % O.BLOCK] = torch.from_numpy(codes)
            pools["cmp_scale"][pg, g % O.BLOCK] = torch.from_numpy(sb)
        for b, g, codes, sb in idx:
            pg = int(table[b, g // O.BLOCK])
            pools["idx_pool"][pg, g % O.BLOCK] = torch.from_numpy(codes)
            pools["idx_kscale"][pg, g % O.BLOCK] = torch.from_numpy(sb)
        return pools, main, idx
    for b, g, vals in main:
        pg = int(table[b, g // O.BLOCK])
        pools["cmp_pool"][pg, g % O.BLOCK] = torch.from_numpy(vals).to(torch.bfloat16)
    for b, g, codes, scale in idx:
        pg = int(table[b, g // O.BLOCK])
        pools["idx_pool"][pg, g % O.BLOCK] = torch.from_numpy(codes)
        pools["idx_scale"][pg, g % O.BLOCK] = float(np.float32(scale))
    return pools, main, idx


def index_row(t, spec, pools, row, relu=True):
    b = int(t["row_req"][row])
    p = int(t["row_pos"][row])
    return O.index_scores(t["q_idx"][row], t["idx_w"][row], p, int(t["n_cmp"][b]), spec.ratio,
                          _idx_pool(t, pools), pools.get("idx_scale"), t["cmp_table"][b].numpy(),
                          relu=relu, rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
                          rope_dim=spec.rope_dim)


def attention_row(t, spec, pools, row, topk_row, inv_rope_out=False, use_sink=True):
    b = int(t["row_req"][row])
    p = int(t["row_pos"][row])
    kv_pool, cmp_pool = _kv_pools(t, pools)
    return O.sparse_attention(t["q"][row], p, topk_row, kv_pool, t["kv_table"][b].numpy(),
                              cmp_pool, t["cmp_table"][b].numpy(),
                              t["sink"] if use_sink else None, 1.0 / np.sqrt(spec.head_dim),
                              window=spec.window, rope_cos=t["rope_cos"],
                              rope_sin=t["rope_sin"], rope_dim=spec.rope_dim,
                              inv_rope_out=inv_rope_out)


def dense_selection(t, spec, row):
    """HCA's candidates: every visible compressed entry, up to the capacity."""
    b = int(t["row_req"][row])
    v = O.visible_count(int(t["row_pos"][row]), spec.ratio, int(t["n_cmp"][b]))
    sel = np.full(spec.topk, -1, dtype=np.int64)
    sel[:min(v, spec.topk)] = np.arange(min(v, spec.topk))
    return sel


def reindex_tensors(t):
    """The reindex layer of a hierarchical workload: the level-one layer's
    caches with the reindex layer's own q, q_idx, idx_w and sink."""
    r = dict(t)
    for k in ("q", "q_idx", "idx_w", "sink"):
        r[k] = t[k + "2"]
    return r


def full_step(t, spec, rows=None, trace=None):
    """Oracle's own chain: compress -> scores -> top-k -> attention for ``rows``
    (HCA: compress -> attention over every visible compressed entry).  With
    the hierarchical indexer (``spec.n_cand``) the level-one layer also
    selects candidate blocks ("DeepSeek V4.1 Flash", hierarchical indexer)
    and a reindex layer follows: its own scores, top-k inside the candidate
    blocks, attention (entries ``cand``, ``scores2``, ``topk2``, ``out2``,
    ``lse2``).  ``trace`` is handed to ``compress_step``."""
    pools, _, _ = compress_step(t, spec, trace=trace)
    rows = range(spec.n_rows) if rows is None else rows
    res = {}
    t2 = reindex_tensors(t) if spec.n_cand else None
    for row in rows:
        if int(t["row_req"][row]) < 0:
            continue
        if spec.dense:
            sel = dense_selection(t, spec, row)
            out, lse = attention_row(t, spec, pools, row, sel)
            res[row] = dict(scores=None, topk=sel, out=out, lse=lse)
            continue
        s = index_row(t, spec, pools, row)
        sel = O.topk_select(s, spec.topk)
        out, lse = attention_row(t, spec, pools, row, sel)
        res[row] = dict(scores=s, topk=sel, out=out, lse=lse)
        if spec.n_cand:
            cand = O.select_blocks(s, spec.n_cand, spec.cand_block)
            s2 = index_row(t2, spec, pools, row)
            sel2 = O.topk_in_blocks(s2, cand, spec.topk, spec.cand_block)
            out2, lse2 = attention_row(t2, spec, pools, row, sel2)
            res[row].update(cand=cand, scores2=s2, topk2=sel2, out2=out2, lse2=lse2)
    return pools, res
