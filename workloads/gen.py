"""Seeded workload generator (inputs only; see the package docstring)."""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 128  # rows per KV page (V4-Flash MTP page, "Deployment configuration")


@dataclass
class WorkloadSpec:
    """Shape of one synthetic CSA step.

    Request b holds ``ctx[b]`` tokens after this step; the step's query rows
    are its last ``chunk[b]`` positions.  ``n_cmp[b] = ctx[b] // ratio``
    compressed entries are published.
    """

    name: str
    ctx: list
    chunk: list
    ratio: int
    topk: int
    seed: int
    mode: str = "decode"  # "decode" or "prefill"
    heads: int = 64
    head_dim: int = 512
    idx_heads: int = 64
    idx_dim: int = 128
    window: int = 128
    rope_dim: int = 64
    theta: float = 10000.0
    rope_cap: int | None = None  # default: next power of two above the largest position
    kv_pool_pages: int | None = None  # default: exactly the pages used
    cmp_pool_pages: int | None = None
    kv_pages: str = "all"  # "all" or "window" (only pages the window reads; others -1)
    cmp_init: str = "random"  # "random" or "zeros" (filled by the compressor)
    pad_rows: int = 0  # trailing padding rows (row_req = -1)
    state: bool = False  # compressors keep a recurrent state ring (capacity max(4, ratio),
    #                      doubled with overlap)
    overlap: bool = False  # overlapping compressors: each entry pools the previous group too
    dense: bool = False  # HCA: no indexer, attention over every visible compressed entry
    # hierarchical indexer: a level-one layer selects n_cand blocks of
    # cand_block compressed positions and a reindex layer (its own q, q_idx,
    # idx_w and sink: q2, q_idx2, idx_w2, sink2) selects inside them; 0 = off
    n_cand: int = 0
    cand_block: int = 8
    # low-bit caches (the production cache ABI of DeepSeek V4.1 Flash): window
    # KV MXFP8 (kv_pool uint8 codes + kv_scale), compressed KV FP4 with E4M3
    # scales (cmp_pool uint8 + cmp_scale), index keys FP4 with E8M0 scales
    # (idx_pool uint8 + idx_kscale)
    lowbit: bool = False
    key_fmt: str = "fp4"  # low-bit index keys: "fp4" (E2M1 + E8M0) or "mxfp8" (E4M3 + E8M0)
    extra: dict = field(default_factory=dict)

    @property
    def n_req(self) -> int:
        return len(self.ctx)

    @property
    def n_rows(self) -> int:
        return int(sum(self.chunk)) + self.pad_rows


CONFIGS = {
    # 1 request, rows at positions 1022 and 1023, ratio 2, top-k 128, table capacity 4096.
    "tiny_decode": WorkloadSpec("tiny_decode", [1024], [2], ratio=2, topk=128, seed=0,
                                rope_cap=4096),
    # 4 requests x 2 rows, contexts 8192/6000/4097/2048, ratio 2, top-k 512,
    # one shared pool of 256 pages each for kv and cmp.
    "serving_decode": WorkloadSpec("serving_decode", [8192, 6000, 4097, 2048], [2, 2, 2, 2],
                                   ratio=2, topk=512, seed=1, kv_pool_pages=256,
                                   cmp_pool_pages=256),
    # 4 requests x 2 rows at 131,072 context, ratio 1, top-k 1024.
    "ratio1_decode": WorkloadSpec("ratio1_decode", [131072] * 4, [2] * 4, ratio=1, topk=1024,
                                  seed=2, kv_pages="window"),
    # 1 request, 8192 tokens at positions 0..8191, ratio 4, top-k 512; the
    # compressor fills cmp_kv and idx_kv in the same step.
    "chunked_prefill": WorkloadSpec("chunked_prefill", [8192], [8192], ratio=4, topk=512, seed=3,
                                    mode="prefill", cmp_init="zeros"),
    # serving_decode's requests at ratio 4 with the compressors' recurrent state
    # rings: each request's group closes on this step's second row and takes
    # its first two tokens from the ring.
    "stateful_decode": WorkloadSpec("stateful_decode", [8192, 6000, 4096, 2048], [2, 2, 2, 2],
                                    ratio=4, topk=512, seed=5, kv_pool_pages=256,
                                    cmp_pool_pages=256, state=True),
    # HCA (ratio 128, dense compressed visibility): an 8192-token prefill chunk
    # whose compressor fills the 64 entries, and a decode step of 4 requests x
    # 2 rows at 131,072 positions whose groups close through the state ring
    # (capacity 128).  top-k is the dense capacity.
    "hca_prefill": WorkloadSpec("hca_prefill", [8192], [8192], ratio=128, topk=64, seed=6,
                                mode="prefill", cmp_init="zeros", dense=True),
    "hca_decode": WorkloadSpec("hca_decode", [131072] * 4, [2] * 4, ratio=128, topk=1024, seed=7,
                               kv_pages="window", dense=True, state=True),
    # 4 requests x 2 rows at 1,048,576 positions, ratio 4, top-k 2048.
    "million_decode": WorkloadSpec("million_decode", [1048576] * 4, [2] * 4, ratio=4, topk=2048,
                                   seed=4, kv_pages="window"),
    # the hierarchical indexer at 1,048,576 positions: a level-one layer (ratio
    # 4, top-k 512) also picks 2,048 blocks of 8 compressed positions; a
    # reindex layer selects its 512 inside them.  4 requests x 2 rows.
    "hier_decode": WorkloadSpec("hier_decode", [1048576] * 4, [2] * 4, ratio=4, topk=512,
                                seed=8, kv_pages="window", n_cand=2048, cand_block=8),
    # serving_decode's requests with the low-bit caches (ratio 2, as the pages'
    # FP4 compressed pools): MXFP8 window, FP4 compressed KV and index keys
    "lowbit_decode": WorkloadSpec("lowbit_decode", [8192, 6000, 4097, 2048], [2, 2, 2, 2],
                                  ratio=2, topk=512, seed=9, kv_pool_pages=256,
                                  cmp_pool_pages=256, lowbit=True),
    # chunked_prefill with the low-bit caches: the compressors publish FP4
    # entries, the indexer reads FP4 keys, the attention its BF16 arena
    "lowbit_prefill": WorkloadSpec("lowbit_prefill", [8192], [8192], ratio=4, topk=512, seed=11,
                                   mode="prefill", cmp_init="zeros", lowbit=True),
    # million_decode with the low-bit caches
    "lowbit_million": WorkloadSpec("lowbit_million", [1048576] * 4, [2] * 4, ratio=4, topk=2048,
                                   seed=10, kv_pages="window", lowbit=True),
    # the overlapping ratio-4 compressors (each entry pools the previous
    # group's four tokens too): stateful_decode's requests with rings of
    # eight slots, and chunked_prefill's 8192-token chunk
    "overlap_decode": WorkloadSpec("overlap_decode", [8192, 6000, 4096, 2048], [2, 2, 2, 2],
                                   ratio=4, topk=512, seed=12, kv_pool_pages=256,
                                   cmp_pool_pages=256, state=True, overlap=True),
    "overlap_prefill": WorkloadSpec("overlap_prefill", [8192], [8192], ratio=4, topk=512, seed=13,
                                    mode="prefill", cmp_init="zeros", overlap=True),
}


def spec_for(name: str, **overrides) -> WorkloadSpec:
    spec = dataclasses.replace(CONFIGS[name])
    return dataclasses.replace(spec, **overrides) if overrides else spec


def _next_pow2_above(x: int) -> int:
    return 1 << int(x).bit_length()


def rope_tables(capacity: int, rope_dim: int = 64, theta: float = 10000.0):
    """FP32 half-width cos/sin tables [capacity, rope_dim // 2] (fixture initialisation)."""
    half = rope_dim // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / rope_dim)
    cos = np.empty((capacity, half), dtype=np.float32)
    sin = np.empty((capacity, half), dtype=np.float32)
    step = 1 << 16
    for p0 in range(0, capacity, step):
        p = np.arange(p0, min(capacity, p0 + step), dtype=np.float64)
        ang = p[:, None] * inv_freq[None, :]
        cos[p0:p0 + len(p)] = np.cos(ang)
        sin[p0:p0 + len(p)] = np.sin(ang)
    return torch.from_numpy(cos), torch.from_numpy(sin)


def _normal_bf16(rng, shape, std=1.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


@dataclass
class Workload:
    spec: WorkloadSpec
    t: dict  # name -> CPU tensor

    def __getattr__(self, k):
        t = self.__dict__.get("t")
        if t is not None and k in t:
            return t[k]
        raise AttributeError(k)

    def to(self, device) -> dict:
        return {k: v.to(device) for k, v in self.t.items()}


def make_workload(spec: WorkloadSpec) -> Workload:
    rng = np.random.default_rng(spec.seed)
    B, r, Dm, Di = spec.n_req, spec.ratio, spec.head_dim, spec.idx_dim
    ctx = [int(c) for c in spec.ctx]
    chunk = [int(c) for c in spec.chunk]
    assert len(chunk) == B and all(0 <= chunk[b] <= ctx[b] for b in range(B))
    n_cmp = [c // r for c in ctx]

    # query rows: the last chunk[b] positions of each request, then padding
    row_req, row_pos = [], []
    for b in range(B):
        for p in range(ctx[b] - chunk[b], ctx[b]):
            row_req.append(b)
            row_pos.append(p)
    row_req += [-1] * spec.pad_rows
    row_pos += [-1] * spec.pad_rows
    T = len(row_req)
    max_pos = max(ctx) - 1
    cap = spec.rope_cap or _next_pow2_above(max_pos)

    # ---- paging: which logical pages exist, then a random physical assignment
    kv_max_blocks = max(1, max(math.ceil(c / BLOCK) for c in ctx))
    cmp_max_blocks = max(1, max(math.ceil(n / BLOCK) for n in n_cmp))
    kv_need = []  # (b, logical page)
    for b in range(B):
        npg = math.ceil(ctx[b] / BLOCK)
        if spec.kv_pages == "window":
            lo = max(0, ctx[b] - chunk[b] - (spec.window - 1))
            pages = range(lo // BLOCK, npg)
        else:
            pages = range(npg)
        kv_need += [(b, j) for j in pages]
    cmp_need = [(b, j) for b in range(B) for j in range(math.ceil(n_cmp[b] / BLOCK))]
    P_kv = spec.kv_pool_pages or max(1, len(kv_need))
    P_c = spec.cmp_pool_pages or max(1, len(cmp_need))
    assert P_kv >= len(kv_need) and P_c >= len(cmp_need)
    kv_perm = rng.permutation(P_kv)
    cmp_perm = rng.permutation(P_c)
    kv_table = np.full((B, kv_max_blocks), -1, dtype=np.int32)
    cmp_table = np.full((B, cmp_max_blocks), -1, dtype=np.int32)
    for i, (b, j) in enumerate(kv_need):
        kv_table[b, j] = kv_perm[i]
    for i, (b, j) in enumerate(cmp_need):
        cmp_table[b, j] = cmp_perm[i]

    # ---- pools
    if spec.lowbit:
        lb = _lowbit_pools(rng, spec, P_kv, P_c)
        kv_pool, cmp_pool, idx_pool = lb["kv_pool"], lb["cmp_pool"], lb["idx_pool"]
        idx_scale = torch.zeros((P_c, BLOCK), dtype=torch.float32)  # unused by FP4 keys
    elif spec.cmp_init == "random":
        kv_pool = _normal_bf16(rng, (P_kv, BLOCK, Dm))
        cmp_pool = _normal_bf16(rng, (P_c, BLOCK, Dm))
        idx_pool = torch.from_numpy(rng.integers(-127, 128, size=(P_c, BLOCK, Di), dtype=np.int8))
        idx_scale = torch.from_numpy(
            rng.uniform(1e-3, 1e-2, size=(P_c, BLOCK)).astype(np.float32))
    else:
        kv_pool = _normal_bf16(rng, (P_kv, BLOCK, Dm))
        cmp_pool = torch.zeros((P_c, BLOCK, Dm), dtype=torch.bfloat16)
        idx_pool = torch.zeros((P_c, BLOCK, Di), dtype=torch.int8)
        idx_scale = torch.zeros((P_c, BLOCK), dtype=torch.float32)

    # ---- per-row activations
    q = _normal_bf16(rng, (T, spec.heads, Dm))
    q_idx = _normal_bf16(rng, (T, spec.idx_heads, Di))
    idx_w = torch.from_numpy(
        (rng.standard_normal((T, spec.idx_heads)) / 8.0).astype(np.float32))
    sink = torch.from_numpy(rng.standard_normal(spec.heads).astype(np.float32))
    # raw KV rows of this chunk are the pool rows at the rows' positions (the
    # window cache holds the same rows); the index compressor gets its own rows
    kv_raw = torch.empty((T, Dm), dtype=torch.bfloat16)
    for t in range(T):
        b, p = row_req[t], row_pos[t]
        if b >= 0 and not spec.lowbit:
            kv_raw[t] = kv_pool[int(kv_table[b, p // BLOCK]), p % BLOCK]
        else:
            kv_raw[t] = _normal_bf16(rng, (Dm,))
    idx_raw = _normal_bf16(rng, (T, Di))
    w_gate = _normal_bf16(rng, (Dm, Dm), std=1.0 / math.sqrt(Dm))
    ape = torch.from_numpy(rng.standard_normal((r, Dm)).astype(np.float32))
    w_gate_i = _normal_bf16(rng, (Di, Di), std=1.0 / math.sqrt(Di))
    ape_i = torch.from_numpy(rng.standard_normal((r, Di)).astype(np.float32))
    rope_cos, rope_sin = rope_tables(cap, spec.rope_dim, spec.theta)

    t = dict(
        row_req=torch.tensor(row_req, dtype=torch.int32),
        row_pos=torch.tensor(row_pos, dtype=torch.int32),
        kv_len=torch.tensor(ctx, dtype=torch.int32),
        n_cmp=torch.tensor(n_cmp, dtype=torch.int32),
        kv_pool=kv_pool,
        kv_table=torch.from_numpy(kv_table),
        cmp_pool=cmp_pool,
        idx_pool=idx_pool,
        idx_scale=idx_scale,
        cmp_table=torch.from_numpy(cmp_table),
        q=q,
        q_idx=q_idx,
        idx_w=idx_w,
        sink=sink,
        kv_raw=kv_raw,
        idx_raw=idx_raw,
        w_gate=w_gate,
        ape=ape,
        w_gate_i=w_gate_i,
        ape_i=ape_i,
        rope_cos=rope_cos,
        rope_sin=rope_sin,
    )
    if spec.state:
        # one ring block per request (plus a spare) in a shuffled order; the
        # slots hold earlier tokens' kv rows (BF16 values) and gate scores
        cap = max(4, r) * (2 if spec.overlap else 1)
        t["state_table"] = torch.from_numpy(rng.permutation(B + 1)[:B].astype(np.int32))
        for name, d in (("state_main", Dm), ("state_idx", Di)):
            kv_part = _normal_bf16(rng, (B + 1, cap, d)).float()
            score_part = torch.from_numpy(
                (rng.standard_normal((B + 1, cap, d)) * 1.4).astype(np.float32))
            t[name] = torch.cat([kv_part, score_part], dim=2).contiguous()
    if spec.lowbit:
        t.update(kv_scale=lb["kv_scale"], cmp_scale=lb["cmp_scale"], idx_kscale=lb["idx_kscale"])
    if spec.n_cand:
        # the reindex layer's own activations and sink
        t["q2"] = _normal_bf16(rng, (T, spec.heads, Dm))
        t["q_idx2"] = _normal_bf16(rng, (T, spec.idx_heads, Di))
        t["idx_w2"] = torch.from_numpy(
            (rng.standard_normal((T, spec.idx_heads)) / 8.0).astype(np.float32))
        t["sink2"] = torch.from_numpy(rng.standard_normal(spec.heads).astype(np.float32))
    return Workload(spec=spec, t=t)


def _lowbit_pools(rng, spec, P_kv, P_c):
    """Random low-bit pools: codes are random bit patterns (no quantisation
    happens here).  Window MXFP8 codes: random sign, E4M3 exponent field 4..8
    and mantissa (magnitudes 1/8 .. 3.75), E8M0 scales 2^-1 or 2^0; FP4
    compressed KV: uniform nibbles, E4M3 scales with exponent field 4..7
    (1/8 .. 1.875); FP4 index keys: uniform nibbles, E8M0 scales 2^-3 .. 2^0;
    FP8 index keys (key_fmt "mxfp8"): E4M3 codes drawn like the window's, the
    same E8M0 scales.
    With ``cmp_init="zeros"`` the compressed pools start as zero bytes (the
    step's compressors fill them)."""
    Dm, Di = spec.head_dim, spec.idx_dim
    shp = (P_kv, BLOCK, Dm)
    kv = (rng.integers(0, 2, shp, dtype=np.uint8) << 7) | (rng.integers(4, 9, shp, dtype=np.uint8) << 3) \
        | rng.integers(0, 8, shp, dtype=np.uint8)
    out = dict(kv_pool=torch.from_numpy(kv.astype(np.uint8)),
               kv_scale=torch.from_numpy(rng.integers(126, 128, (P_kv, BLOCK, Dm // 32),
                                                      dtype=np.uint8)))
    if spec.cmp_init == "random":
        g = (P_c, BLOCK, Dm // 16)
        out["cmp_pool"] = torch.from_numpy(rng.integers(0, 256, (P_c, BLOCK, Dm // 2), dtype=np.uint8))
        out["cmp_scale"] = torch.from_numpy(
            ((rng.integers(4, 8, g, dtype=np.uint8) << 3) | rng.integers(0, 8, g, dtype=np.uint8))
            .astype(np.uint8))
        if spec.key_fmt == "mxfp8":  # E4M3 codes drawn like the window's
            ks = (P_c, BLOCK, Di)
            out["idx_pool"] = torch.from_numpy(
                ((rng.integers(0, 2, ks, dtype=np.uint8) << 7) |
                 (rng.integers(4, 9, ks, dtype=np.uint8) << 3) |
                 rng.integers(0, 8, ks, dtype=np.uint8)).astype(np.uint8))
        else:
            out["idx_pool"] = torch.from_numpy(
                rng.integers(0, 256, (P_c, BLOCK, Di // 2), dtype=np.uint8))
        out["idx_kscale"] = torch.from_numpy(rng.integers(124, 128, (P_c, BLOCK, Di // 32),
                                                          dtype=np.uint8))
    else:
        out["cmp_pool"] = torch.zeros((P_c, BLOCK, Dm // 2), dtype=torch.uint8)
        out["cmp_scale"] = torch.zeros((P_c, BLOCK, Dm // 16), dtype=torch.uint8)
        out["idx_pool"] = torch.zeros((P_c, BLOCK, Di if spec.key_fmt == "mxfp8" else Di // 2),
                                      dtype=torch.uint8)
        out["idx_kscale"] = torch.zeros((P_c, BLOCK, Di // 32), dtype=torch.uint8)
    return out


def reindex_view(t: dict) -> dict:
    """The tensors of the reindex layer: the level-one layer's caches and
    tables with the reindex layer's own q, q_idx, idx_w and sink."""
    r = dict(t)
    for k in ("q", "q_idx", "idx_w", "sink"):
        r[k] = t[k + "2"]
    return r


def random_selection(limits, k, seed):
    """Seeded selections for feeding the attention call directly: for row t,
    min(k, limits[t]) distinct integers drawn uniformly from [0, limits[t]),
    in ascending order, padded with -1 (an input, not a computed top-k)."""
    rng = np.random.default_rng(seed)
    out = np.full((len(limits), k), -1, dtype=np.int32)
    for t, lim in enumerate(limits):
        lim = int(lim)
        if lim <= 0:
            continue
        m = min(k, lim)
        out[t, :m] = np.sort(rng.choice(lim, size=m, replace=False))
    return torch.from_numpy(out)
