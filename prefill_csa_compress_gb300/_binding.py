"""ctypes binding of ``libcsa.so`` (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module only checks
tensor dtypes and devices, fills the C argument structs declared in
``include/csa.h``, sizes the caller-side workspace with torch, and raises
when the library reports an error.  Importing it never builds anything; a
missing library raises ``RuntimeError`` at first use.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_size_t, c_uint32, c_uint64, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa.so")

CSA_OK, CSA_ERR_INVALID_ARG, CSA_ERR_UNSUPPORTED, CSA_ERR_CUDA, CSA_ERR_TIMEOUT = range(5)
CSA_DEV_BAD_BLOCK, CSA_DEV_BAD_POS, CSA_DEV_BAD_INDEX, CSA_DEV_POS_GE_CAP, CSA_DEV_TIMEOUT = (
    0x1, 0x2, 0x4, 0x8, 0x10)
CSA_OUT_BF16, CSA_OUT_INT8 = 0, 1
CSA_FMT_BF16, CSA_FMT_INT8, CSA_FMT_FP4_E4M3, CSA_FMT_FP4_E8M0, CSA_FMT_MXFP8 = 0, 1, 2, 3, 4
CSA_MODE_AUTO, CSA_MODE_DECODE, CSA_MODE_PREFILL = 0, 1, 2
KERNEL_IDS = {
    "compress_gate": 0, "compress_pool": 1, "compress_fused": 2, "index_score": 3,
    "index_topk": 4, "attn_decode": 5, "attn_prefill": 6, "dequant": 7,
}


class CsaError(RuntimeError):
    def __init__(self, call, status):
        super().__init__(f"{call} failed: status {status} ({status_string(status)})")
        self.status = status


class CompressArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", c_uint32), ("n_rows", c_int32), ("ratio", c_int32), ("dx", c_int32),
        ("d", c_int32), ("out_mode", c_int32), ("rotate", c_int32), ("rope_cap", c_int32),
        ("x", c_void_p), ("kv", c_void_p), ("w_gate", c_void_p), ("ape", c_void_p),
        ("gamma", c_void_p), ("rms_eps", c_float), ("positions", c_void_p),
        ("row_req", c_void_p), ("rope_cos", c_void_p), ("rope_sin", c_void_p),
        ("block_table", c_void_p), ("n_req", c_int32), ("max_blocks", c_int32),
        ("n_blocks", c_int32), ("cmp_pool", c_void_p), ("idx_pool", c_void_p),
        ("idx_scale_pool", c_void_p), ("status_dev", c_void_p), ("workspace", c_void_p),
        ("workspace_bytes", c_size_t), ("state_cache", c_void_p),
        ("state_block_table", c_void_p), ("n_state_blocks", c_int32),
        ("state_capacity", c_int32), ("scale_pool", c_void_p), ("overlap", c_int32),
        ("pool_page_stride", ctypes.c_int64), ("pool_row_stride", ctypes.c_int64),
        ("scale_page_stride", ctypes.c_int64),
    ]


class IndexArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", c_uint32), ("n_rows", c_int32), ("n_heads", c_int32),
        ("head_dim", c_int32), ("ratio", c_int32), ("topk", c_int32), ("relu", c_int32),
        ("mode", c_int32), ("q_idx", c_void_p), ("weights", c_void_p), ("row_req", c_void_p),
        ("row_pos", c_void_p), ("n_cmp", c_void_p), ("idx_pool", c_void_p),
        ("idx_scale_pool", c_void_p), ("cmp_block_table", c_void_p), ("n_req", c_int32),
        ("max_blocks", c_int32), ("n_blocks", c_int32), ("rope_cos", c_void_p),
        ("rope_sin", c_void_p), ("rope_cap", c_int32), ("topk_idx", c_void_p),
        ("topk_score", c_void_p), ("scores", c_void_p), ("score_cols", c_int32),
        ("status_dev", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("cand_block", c_int32), ("n_cand", c_int32), ("cand_out", c_void_p),
        ("cand_in", c_void_p), ("key_fmt", c_int32), ("key_scale_pool", c_void_p),
        ("wait_limit_ns", ctypes.c_int64), ("key_page_stride", ctypes.c_int64),
        ("key_row_stride", ctypes.c_int64), ("scale_page_stride", ctypes.c_int64),
    ]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", c_uint32), ("n_rows", c_int32), ("n_heads", c_int32),
        ("head_dim", c_int32), ("ratio", c_int32), ("topk", c_int32), ("window", c_int32),
        ("inv_rope_out", c_int32), ("softmax_scale", c_float), ("q", c_void_p),
        ("row_req", c_void_p), ("row_pos", c_void_p), ("topk_idx", c_void_p),
        ("kv_pool", c_void_p), ("kv_block_table", c_void_p), ("kv_max_blocks", c_int32),
        ("kv_n_blocks", c_int32), ("kv_len", c_void_p), ("cmp_pool", c_void_p),
        ("cmp_block_table", c_void_p), ("cmp_max_blocks", c_int32), ("cmp_n_blocks", c_int32),
        ("n_cmp", c_void_p), ("n_req", c_int32), ("sink", c_void_p), ("rope_cos", c_void_p),
        ("rope_sin", c_void_p), ("rope_cap", c_int32), ("out", c_void_p), ("lse", c_void_p),
        ("status_dev", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("kv_fmt", c_int32), ("cmp_fmt", c_int32), ("kv_scale_pool", c_void_p),
        ("cmp_scale_pool", c_void_p), ("kv_page_stride", ctypes.c_int64),
        ("kv_row_stride", ctypes.c_int64), ("cmp_page_stride", ctypes.c_int64),
        ("cmp_row_stride", ctypes.c_int64),
    ]


_lib = None


def lib():
    """The loaded ``libcsa.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (the CSA path has no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, argt in (("csa_compress", CompressArgs), ("csa_index_topk", IndexArgs),
                           ("csa_index_topk_noalloc", IndexArgs),
                           ("csa_sparse_attn_decode", AttnArgs),
                           ("csa_sparse_attn_prefill", AttnArgs)):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(argt), c_void_p]
            f.restype = c_int32
        L.csa_compress_pair.argtypes = [ctypes.POINTER(CompressArgs), ctypes.POINTER(CompressArgs),
                                        c_void_p]
        L.csa_compress_pair.restype = c_int32
        L.csa_version.restype = ctypes.c_char_p
        L.csa_status_string.argtypes = [c_int32]
        L.csa_status_string.restype = ctypes.c_char_p
        L.csa_launch_count.restype = c_uint64
        L.csa_prof_enable.argtypes = [c_int32, c_int32]
        L.csa_prof_enable.restype = c_int32
        L.csa_prof_read.argtypes = [c_int32, ctypes.POINTER(c_float), ctypes.POINTER(c_int32)]
        L.csa_prof_read.restype = c_int32
        L.csa_prof_disable.restype = c_int32
        L.csa_prof_join.argtypes = [c_void_p]
        L.csa_prof_join.restype = c_int32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().csa_status_string(int(status)).decode()


def version() -> str:
    return lib().csa_version().decode()


def launch_count() -> int:
    return int(lib().csa_launch_count())


_prof_on = False


def prof_enable(kernel: str, max_launches: int) -> None:
    global _prof_on
    st = lib().csa_prof_enable(KERNEL_IDS[kernel], int(max_launches))
    if st != CSA_OK:
        raise CsaError("csa_prof_enable", st)
    _prof_on = True


def prof_join(stream=None) -> None:
    """Bring the timing events' side stream back into ``stream`` (needed
    before a stream capture that recorded timed launches ends)."""
    if not _prof_on:
        return
    st = lib().csa_prof_join(_stream(stream))
    if st != CSA_OK:
        raise CsaError("csa_prof_join", st)


def prof_read(kernel: str):
    ms, n = c_float(0.0), c_int32(0)
    st = lib().csa_prof_read(KERNEL_IDS[kernel], ctypes.byref(ms), ctypes.byref(n))
    if st != CSA_OK:
        raise CsaError("csa_prof_read", st)
    return float(ms.value), int(n.value)


def prof_disable() -> None:
    global _prof_on
    lib().csa_prof_disable()
    _prof_on = False


# ---------------------------------------------------------------- marshalling helpers


def _shape(t, want, name):
    """Checks a tensor's shape (None matches any size)."""
    if t is None or t.dim() != len(want) or any(w is not None and int(g) != w
                                                   for g, w in zip(t.shape, want)):
        raise ValueError(f"{name} must have shape {want}, got "
                         f"{None if t is None else tuple(t.shape)}")


def _p(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _pool(t, dtype, name):
    """A paged pool [pages, 128, ...] that may be a view into a larger
    allocation: its pointer and its page and row strides in bytes (each row's
    own elements contiguous).  A scale pool [pages, 128] must have
    contiguous rows.  Returns (pointer, page stride, row stride)."""
    if t is None:
        return None, 0, 0
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() < 2 or t.shape[1] != 128:
        raise ValueError(f"{name} must be [pages, 128, ...]")
    inner = t[0, 0] if t.shape[0] else t
    if t.shape[0] and t.dim() > 2 and not inner.is_contiguous():
        raise ValueError(f"{name}: a row's elements must be contiguous")
    es = t.element_size()
    if t.dim() == 2:
        if t.stride(1) != 1:
            raise ValueError(f"{name}: a page's entries must be contiguous")
        return t.data_ptr(), t.stride(0) * es, es
    return t.data_ptr(), t.stride(0) * es, t.stride(1) * es


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return c_void_p(s.cuda_stream)


class PreparedCall:
    """A fully marshalled library call: the argument struct and workspace are
    built once; calling it only crosses the C ABI (for repeated steps)."""

    def __init__(self, fn_name, args, workspace):
        self.fn_name = fn_name
        self.fn = getattr(lib(), fn_name)
        self.args = args if isinstance(args, tuple) else (args,)
        self.workspace = workspace
        self._refs = tuple(ctypes.byref(a) for a in self.args)

    def __call__(self, stream=None):
        st = self.fn(*self._refs, _stream(stream))
        if st != CSA_OK:
            raise CsaError(self.fn_name, st)
        return self.workspace


def _run(fn_name, args, workspace, stream, device, prepare=False):
    fn = getattr(lib(), fn_name)
    args.workspace = None
    args.workspace_bytes = 0
    st = fn(ctypes.byref(args), None)  # size query
    if st != CSA_OK:
        raise CsaError(fn_name, st)
    need = int(args.workspace_bytes)
    if workspace is None or workspace.numel() < need:
        # zero-filled: the decode attention's split counters must start at zero
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
    args.workspace = workspace.data_ptr()
    args.workspace_bytes = workspace.numel()
    call = PreparedCall(fn_name, args, workspace)
    if prepare:
        return call
    return call(stream)


def _fill_common_rope(args, rope_cos, rope_sin):
    """FP32 half-width tables; capacity = table rows."""
    args.rope_cos = _p(rope_cos, torch.float32, "rope_cos")
    args.rope_sin = _p(rope_sin, torch.float32, "rope_sin")
    args.rope_cap = int(rope_cos.shape[0]) if rope_cos is not None else 0


# ---------------------------------------------------------------- the four calls


_OUT_MODES = {"bf16": 0, "int8": 1, "fp4_e4m3": 2, "fp4_e8m0": 3, "mxfp8": 4}


def _compress_struct(*, x, kv, w_gate, ape, ratio, positions, row_req, block_table, out="bf16",
                     cmp_pool=None, idx_pool=None, idx_scale_pool=None, scale_pool=None,
                     gamma=None, rms_eps=1e-6, rotate=False, rope_cos=None, rope_sin=None,
                     status=None, state_cache=None, state_block_table=None, overlap=False):
    a = CompressArgs()
    a.struct_size = ctypes.sizeof(CompressArgs)
    a.n_rows = int(x.shape[0])
    a.ratio = int(ratio)
    a.dx = int(x.shape[1])
    a.d = int(kv.shape[1])
    a.out_mode = _OUT_MODES[out]
    a.rotate = 1 if rotate else 0
    a.overlap = 1 if overlap else 0
    a.x = _p(x, torch.bfloat16, "x")
    a.kv = _p(kv, torch.bfloat16, "kv")
    a.w_gate = _p(w_gate, torch.bfloat16, "w_gate")
    a.ape = _p(ape, torch.float32, "ape")
    a.gamma = _p(gamma, torch.bfloat16, "gamma")
    a.rms_eps = float(rms_eps)
    a.positions = _p(positions, torch.int32, "positions")
    a.row_req = _p(row_req, torch.int32, "row_req")
    _fill_common_rope(a, rope_cos, rope_sin)
    a.block_table = _p(block_table, torch.int32, "block_table")
    a.n_req, a.max_blocks = int(block_table.shape[0]), int(block_table.shape[1])
    if a.out_mode == CSA_OUT_BF16:
        a.cmp_pool, a.pool_page_stride, a.pool_row_stride = _pool(cmp_pool, torch.bfloat16,
                                                                  "cmp_pool")
        a.n_blocks = int(cmp_pool.shape[0])
    elif out in ("fp4_e4m3", "fp4_e8m0", "mxfp8"):  # codes into cmp_pool, scales into scale_pool
        group = 16 if out == "fp4_e4m3" else 32
        _shape(cmp_pool, (None, 128, a.d if out == "mxfp8" else a.d // 2), "cmp_pool")
        _shape(scale_pool, (cmp_pool.shape[0], 128, a.d // group), "scale_pool")
        a.cmp_pool = _p(cmp_pool, torch.uint8, "cmp_pool")
        a.scale_pool = _p(scale_pool, torch.uint8, "scale_pool")
        a.n_blocks = int(cmp_pool.shape[0])
    else:
        a.idx_pool, a.pool_page_stride, a.pool_row_stride = _pool(idx_pool, torch.int8,
                                                                  "idx_pool")
        a.idx_scale_pool, a.scale_page_stride, _ = _pool(idx_scale_pool, torch.float32,
                                                         "idx_scale_pool")
        a.n_blocks = int(idx_pool.shape[0])
    a.status_dev = _p(status, torch.int32, "status")
    if state_cache is not None:
        a.state_cache = _p(state_cache, torch.float32, "state_cache")
        a.state_block_table = _p(state_block_table, torch.int32, "state_block_table")
        a.n_state_blocks, a.state_capacity = int(state_cache.shape[0]), int(state_cache.shape[1])
    return a


def csa_compress(*, workspace=None, stream=None, prepare=False, **kw):
    """Gated compression of the chunk's complete groups into a paged pool
    (``include/csa.h``: csa_compress).  Keywords: x, kv, w_gate, ape, ratio,
    positions, row_req, block_table, out ("bf16", "int8", "fp4_e4m3" or
    "fp4_e8m0"), cmp_pool (bf16; uint8 codes for fp4 with scale_pool) or
    idx_pool + idx_scale_pool, gamma, rms_eps, rotate, rope_cos, rope_sin,
    status, and for the recurrent state ring state_cache (FP32 [blocks,
    capacity, 2 d]) with state_block_table (INT32 [n_req]); ``overlap`` pools
    each entry over the previous group's tokens too."""
    a = _compress_struct(**kw)
    return _run("csa_compress", a, workspace, stream, kw["x"].device, prepare)


def csa_compress_pair(first: dict, second: dict, *, workspaces=(None, None), stream=None,
                      prepare=False):
    """Two compressors of one layer in one call (``include/csa.h``:
    csa_compress_pair); ``first`` and ``second`` hold csa_compress's keywords.
    Returns the two workspaces (or the prepared call)."""
    structs, wss = [], []
    for kw, ws in zip((first, second), workspaces):
        a = _compress_struct(**kw)
        a.workspace, a.workspace_bytes = None, 0
        st = lib().csa_compress(ctypes.byref(a), None)  # size query
        if st != CSA_OK:
            raise CsaError("csa_compress_pair", st)
        need = int(a.workspace_bytes)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=kw["x"].device)
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        structs.append(a)
        wss.append(ws)
    call = PreparedCall("csa_compress_pair", tuple(structs), tuple(wss))
    if prepare:
        return call
    return call(stream)


def csa_index_topk(*, q_idx, weights, row_req, row_pos, n_cmp, ratio, idx_pool, idx_scale_pool,
                   cmp_block_table, topk, topk_idx, topk_score=None, scores=None, relu=True,
                   rope_cos=None, rope_sin=None, mode=CSA_MODE_AUTO, status=None,
                   cand_out=None, cand_in=None, cand_block=8, key_scale_pool=None,
                   key_fmt="fp4", wait_limit_ns=0, workspace=None, stream=None,
                   prepare=False):
    """Indexer scores and deterministic top-k (``include/csa.h``: csa_index_topk).

    ``cand_out`` (i32 [n_rows, n_cand]) also selects the level-one candidate
    blocks; ``cand_in`` restricts scoring and selection to given candidate
    blocks (reindex).  With ``key_scale_pool`` (uint8 [blocks, 128, 4]) the
    keys are low-bit, ``key_fmt`` "fp4" (``idx_pool`` uint8 [blocks, 128, 64]:
    packed E2M1 with E8M0 scales per 32 dims) or "mxfp8" (uint8 [blocks, 128,
    128]: E4M3 with E8M0 scales per 32 dims), and ``idx_scale_pool`` is
    unused.  ``wait_limit_ns`` bounds the cooperative top-k's barrier waits
    (0: the library's default)."""
    a = IndexArgs()
    a.struct_size = ctypes.sizeof(IndexArgs)
    a.n_rows = int(q_idx.shape[0])
    a.n_heads = int(q_idx.shape[1])
    a.head_dim = int(q_idx.shape[2])
    a.ratio = int(ratio)
    a.topk = int(topk)
    a.relu = 1 if relu else 0
    a.mode = int(mode)
    a.q_idx = _p(q_idx, torch.bfloat16, "q_idx")
    a.weights = _p(weights, torch.float32, "weights")
    a.row_req = _p(row_req, torch.int32, "row_req")
    a.row_pos = _p(row_pos, torch.int32, "row_pos")
    a.n_cmp = _p(n_cmp, torch.int32, "n_cmp")
    if key_scale_pool is not None:
        _shape(idx_pool, (None, 128, 64 if key_fmt == "fp4" else 128), "idx_pool")
        _shape(key_scale_pool, (idx_pool.shape[0], 128, 4), "key_scale_pool")
        a.key_fmt = CSA_FMT_FP4_E8M0 if key_fmt == "fp4" else CSA_FMT_MXFP8
        a.idx_pool = _p(idx_pool, torch.uint8, "idx_pool")
        a.key_scale_pool = _p(key_scale_pool, torch.uint8, "key_scale_pool")
    else:
        a.key_fmt = CSA_FMT_INT8
        a.idx_pool, a.key_page_stride, a.key_row_stride = _pool(idx_pool, torch.int8, "idx_pool")
        a.idx_scale_pool, a.scale_page_stride, _ = _pool(idx_scale_pool, torch.float32,
                                                         "idx_scale_pool")
    a.cmp_block_table = _p(cmp_block_table, torch.int32, "cmp_block_table")
    a.n_req, a.max_blocks = int(cmp_block_table.shape[0]), int(cmp_block_table.shape[1])
    a.n_blocks = int(idx_pool.shape[0])
    _fill_common_rope(a, rope_cos, rope_sin)
    a.topk_idx = _p(topk_idx, torch.int32, "topk_idx")
    a.topk_score = _p(topk_score, torch.float32, "topk_score")
    a.scores = _p(scores, torch.float32, "scores")
    a.score_cols = int(scores.shape[1]) if scores is not None else 0
    a.status_dev = _p(status, torch.int32, "status")
    a.wait_limit_ns = int(wait_limit_ns)
    cand = cand_out if cand_out is not None else cand_in
    if cand is not None:
        a.cand_block = int(cand_block)
        a.n_cand = int(cand.shape[1])
        a.cand_out = _p(cand_out, torch.int32, "cand_out")
        a.cand_in = _p(cand_in, torch.int32, "cand_in")
    return _run("csa_index_topk", a, workspace, stream, q_idx.device, prepare)


def csa_index_topk_noalloc(*, q_idx, weights, row_req, row_pos, n_cmp, ratio, idx_pool,
                           idx_scale_pool, cmp_block_table, topk, topk_idx, topk_score=None,
                           scores=None, relu=True, rope_cos=None, rope_sin=None,
                           mode=CSA_MODE_AUTO, status=None, stream=None):
    """csa_index_topk without a caller workspace: the library's own score
    scratch is used (``include/csa.h``: csa_index_topk_noalloc)."""
    a = IndexArgs()
    a.struct_size = ctypes.sizeof(IndexArgs)
    a.n_rows, a.n_heads, a.head_dim = (int(x) for x in q_idx.shape)
    a.ratio, a.topk, a.relu, a.mode = int(ratio), int(topk), 1 if relu else 0, int(mode)
    a.q_idx = _p(q_idx, torch.bfloat16, "q_idx")
    a.weights = _p(weights, torch.float32, "weights")
    a.row_req = _p(row_req, torch.int32, "row_req")
    a.row_pos = _p(row_pos, torch.int32, "row_pos")
    a.n_cmp = _p(n_cmp, torch.int32, "n_cmp")
    a.idx_pool = _p(idx_pool, torch.int8, "idx_pool")
    a.idx_scale_pool = _p(idx_scale_pool, torch.float32, "idx_scale_pool")
    a.cmp_block_table = _p(cmp_block_table, torch.int32, "cmp_block_table")
    a.n_req, a.max_blocks = int(cmp_block_table.shape[0]), int(cmp_block_table.shape[1])
    a.n_blocks = int(idx_pool.shape[0])
    _fill_common_rope(a, rope_cos, rope_sin)
    a.topk_idx = _p(topk_idx, torch.int32, "topk_idx")
    a.topk_score = _p(topk_score, torch.float32, "topk_score")
    a.scores = _p(scores, torch.float32, "scores")
    a.score_cols = int(scores.shape[1]) if scores is not None else 0
    a.status_dev = _p(status, torch.int32, "status")
    st = lib().csa_index_topk_noalloc(ctypes.byref(a), _stream(stream))
    if st != CSA_OK:
        raise CsaError("csa_index_topk_noalloc", st)


def _attn(fn_name, *, q, row_req, row_pos, topk_idx, kv_pool, kv_block_table, kv_len, cmp_pool,
          cmp_block_table, n_cmp, ratio, out, lse=None, sink=None, softmax_scale=None,
          window=128, rope_cos=None, rope_sin=None, inv_rope_out=False, status=None,
          workspace=None, stream=None, prepare=False, dense_cap=0, kv_scale_pool=None,
          cmp_scale_pool=None):
    """``topk_idx=None`` with ``dense_cap > 0``: every visible compressed entry
    (up to dense_cap) is a candidate (dense visibility, HCA).  With
    ``kv_scale_pool`` the window pool is MXFP8 (uint8 [blocks, 128, 512] codes,
    uint8 [blocks, 128, 16] scales); with ``cmp_scale_pool`` the compressed
    pool is FP4 (uint8 [blocks, 128, 256] codes, [blocks, 128, 32] E4M3
    scales)."""
    a = AttnArgs()
    a.struct_size = ctypes.sizeof(AttnArgs)
    a.n_rows = int(q.shape[0])
    a.n_heads = int(q.shape[1])
    a.head_dim = int(q.shape[2])
    a.ratio = int(ratio)
    a.topk = int(topk_idx.shape[1]) if topk_idx is not None else int(dense_cap)
    a.window = int(window)
    a.inv_rope_out = 1 if inv_rope_out else 0
    a.softmax_scale = float(softmax_scale if softmax_scale is not None else q.shape[2] ** -0.5)
    a.q = _p(q, torch.bfloat16, "q")
    a.row_req = _p(row_req, torch.int32, "row_req")
    a.row_pos = _p(row_pos, torch.int32, "row_pos")
    a.topk_idx = _p(topk_idx, torch.int32, "topk_idx")
    kv_lb, cmp_lb = kv_scale_pool is not None, cmp_scale_pool is not None
    if kv_lb:
        _shape(kv_pool, (None, 128, 512), "kv_pool")
        _shape(kv_scale_pool, (kv_pool.shape[0], 128, 16), "kv_scale_pool")
    if cmp_lb:
        _shape(cmp_pool, (None, 128, 256), "cmp_pool")
        _shape(cmp_scale_pool, (cmp_pool.shape[0], 128, 32), "cmp_scale_pool")
    a.kv_fmt = CSA_FMT_MXFP8 if kv_lb else CSA_FMT_BF16
    a.cmp_fmt = CSA_FMT_FP4_E4M3 if cmp_lb else CSA_FMT_BF16
    a.kv_scale_pool = _p(kv_scale_pool, torch.uint8, "kv_scale_pool")
    a.cmp_scale_pool = _p(cmp_scale_pool, torch.uint8, "cmp_scale_pool")
    if kv_lb:
        a.kv_pool = _p(kv_pool, torch.uint8, "kv_pool")
    else:  # BF16 pools may be strided views
        a.kv_pool, a.kv_page_stride, a.kv_row_stride = _pool(kv_pool, torch.bfloat16, "kv_pool")
    a.kv_block_table = _p(kv_block_table, torch.int32, "kv_block_table")
    a.kv_max_blocks = int(kv_block_table.shape[1])
    a.kv_n_blocks = int(kv_pool.shape[0])
    a.kv_len = _p(kv_len, torch.int32, "kv_len")
    if cmp_lb:
        a.cmp_pool = _p(cmp_pool, torch.uint8, "cmp_pool")
    else:
        a.cmp_pool, a.cmp_page_stride, a.cmp_row_stride = _pool(cmp_pool, torch.bfloat16,
                                                                "cmp_pool")
    a.cmp_block_table = _p(cmp_block_table, torch.int32, "cmp_block_table")
    a.cmp_max_blocks = int(cmp_block_table.shape[1])
    a.cmp_n_blocks = int(cmp_pool.shape[0])
    a.n_cmp = _p(n_cmp, torch.int32, "n_cmp")
    a.n_req = int(kv_block_table.shape[0])
    a.sink = _p(sink, torch.float32, "sink")
    _fill_common_rope(a, rope_cos, rope_sin)
    a.out = _p(out, torch.bfloat16, "out")
    a.lse = _p(lse, torch.float32, "lse")
    a.status_dev = _p(status, torch.int32, "status")
    return _run(fn_name, a, workspace, stream, q.device, prepare)


def csa_sparse_attn_decode(**kw):
    """Split-K shared-KV sparse attention with sink (``include/csa.h``)."""
    return _attn("csa_sparse_attn_decode", **kw)


def csa_sparse_attn_prefill(**kw):
    """Shared-KV sparse attention with sink, tiled for many rows (``include/csa.h``)."""
    return _attn("csa_sparse_attn_prefill", **kw)
