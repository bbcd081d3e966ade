"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol ``include/csa.h`` declares, the ctypes structs match the C layout, and
argument validation / workspace queries answer without touching the device."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def L():
    from prefill_csa_compress_gb300 import build as B

    B.build()
    from prefill_csa_compress_gb300 import _binding

    return _binding.lib()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"CSA_API\s+[\w\s\*]+?\b(csa_\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"csa_compress", "csa_index_topk", "csa_sparse_attn_decode",
            "csa_sparse_attn_prefill"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in csa.h but not exported"


def test_version_and_status_strings(L):
    from prefill_csa_compress_gb300 import _binding as b

    assert "sm_103a" in b.version()
    assert b.status_string(0) == "ok"
    assert b.status_string(2) == "unsupported shape"


def _c_layout(struct, fields):
    prog = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(){",
            f'printf("%zu\\n", sizeof({struct}));']
    prog += [f'printf("%zu\\n", offsetof({struct}, {f}));' for f in fields]
    prog.append("return 0;}")
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(c, "w").write("\n".join(prog))
        subprocess.check_call(["gcc", c, "-o", exe])
        return [int(x) for x in subprocess.check_output([exe]).split()]


@pytest.mark.parametrize("cname,pyname", [("csa_compress_args", "CompressArgs"),
                                          ("csa_index_args", "IndexArgs"),
                                          ("csa_attn_args", "AttnArgs")])
def test_ctypes_layout_matches_c(cname, pyname):
    from prefill_csa_compress_gb300 import _binding as b

    S = getattr(b, pyname)
    fields = [f for f, _ in S._fields_]
    got = _c_layout(cname, fields)
    assert got[0] == ctypes.sizeof(S)
    for f, off in zip(fields, got[1:]):
        assert getattr(S, f).offset == off, f


def _compress_args(b, **kw):
    a = b.CompressArgs()
    a.struct_size = ctypes.sizeof(a)
    a.n_rows, a.ratio, a.dx, a.d = 8192, 4, 512, 512
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_workspace_queries_and_validation(L):
    from prefill_csa_compress_gb300 import _binding as b

    a = _compress_args(b)
    assert L.csa_compress(ctypes.byref(a), None) == b.CSA_OK
    assert a.workspace_bytes == 8192 * 512 * 4
    assert L.csa_compress(ctypes.byref(_compress_args(b, ratio=3)), None) == b.CSA_ERR_UNSUPPORTED
    assert L.csa_compress(ctypes.byref(_compress_args(b, d=256)), None) == b.CSA_ERR_UNSUPPORTED
    bad = _compress_args(b)
    bad.struct_size = 8
    assert L.csa_compress(ctypes.byref(bad), None) == b.CSA_ERR_INVALID_ARG
    # a real workspace but no tensors: rejected on the host before any launch
    dummy = ctypes.create_string_buffer(256)
    a = _compress_args(b, n_rows=1, workspace=ctypes.addressof(dummy), workspace_bytes=256)
    assert L.csa_compress(ctypes.byref(a), None) == b.CSA_ERR_INVALID_ARG
    assert L.csa_compress(None, None) == b.CSA_ERR_INVALID_ARG
    # the pair: both structs size-queried, either one's error returned
    a1, a2 = _compress_args(b), _compress_args(b, d=128)
    assert L.csa_compress_pair(ctypes.byref(a1), ctypes.byref(a2), None) == b.CSA_OK
    assert (a1.workspace_bytes, a2.workspace_bytes) == (8192 * 512 * 4, 8192 * 128 * 4)
    assert L.csa_compress_pair(ctypes.byref(_compress_args(b)),
                               ctypes.byref(_compress_args(b, ratio=3)), None) == b.CSA_ERR_UNSUPPORTED
    assert L.csa_compress_pair(ctypes.byref(bad), ctypes.byref(_compress_args(b)),
                               None) == b.CSA_ERR_INVALID_ARG
    a = _compress_args(b, n_rows=1, workspace=ctypes.addressof(dummy), workspace_bytes=256)
    a2 = _compress_args(b, n_rows=1, workspace=ctypes.addressof(dummy), workspace_bytes=256)
    assert L.csa_compress_pair(ctypes.byref(a), ctypes.byref(a2), None) == b.CSA_ERR_INVALID_ARG
    assert L.csa_compress_pair(None, ctypes.byref(a2), None) == b.CSA_ERR_INVALID_ARG
    # a caller built without the state-ring fields (smaller struct_size) is accepted
    old = _compress_args(b)
    old.struct_size = b.CompressArgs.state_cache.offset
    assert L.csa_compress(ctypes.byref(old), None) == b.CSA_OK
    assert old.workspace_bytes == 8192 * 512 * 4
    old.struct_size = b.CompressArgs.state_cache.offset - 8
    assert L.csa_compress(ctypes.byref(old), None) == b.CSA_ERR_INVALID_ARG
    # overlap: 0 or 1, ratio <= 64; a struct that ends before `overlap` means 0
    assert L.csa_compress(ctypes.byref(_compress_args(b, overlap=1)), None) == b.CSA_OK
    assert L.csa_compress(ctypes.byref(_compress_args(b, overlap=2)),
                          None) == b.CSA_ERR_INVALID_ARG
    assert L.csa_compress(ctypes.byref(_compress_args(b, overlap=1, ratio=128)),
                          None) == b.CSA_ERR_UNSUPPORTED
    short = _compress_args(b, overlap=1, ratio=128)
    short.struct_size = b.CompressArgs.overlap.offset
    assert L.csa_compress(ctypes.byref(short), None) == b.CSA_OK
    # with overlap the ring needs 2 * ratio slots: checked before any launch
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    ptrs = dict(x=base, kv=base, w_gate=base, ape=base, positions=base, row_req=base,
                block_table=base, cmp_pool=base, n_req=1, max_blocks=1, n_blocks=1,
                workspace=base, workspace_bytes=1 << 14, state_cache=base,
                state_block_table=base, n_state_blocks=1)
    ring = _compress_args(b, n_rows=1, overlap=1, state_capacity=4, **ptrs)
    assert L.csa_compress(ctypes.byref(ring), None) == b.CSA_ERR_INVALID_ARG
    # a state ring needs its table and at least `ratio` slots
    st = ctypes.create_string_buffer(4096)
    ring = _compress_args(b, n_rows=1, workspace=ctypes.addressof(dummy), workspace_bytes=256,
                          state_cache=ctypes.addressof(st), n_state_blocks=1, state_capacity=4)
    assert L.csa_compress(ctypes.byref(ring), None) == b.CSA_ERR_INVALID_ARG  # no tensors, no table

    ia = b.IndexArgs()
    ia.struct_size = ctypes.sizeof(ia)
    ia.n_rows, ia.n_heads, ia.head_dim, ia.ratio, ia.topk, ia.max_blocks = 8, 64, 128, 4, 2048, 2048
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_OK
    # scores (8 rows x 262144 FP32) plus the multi-CTA top-k scratch
    assert ia.workspace_bytes > 8 * 2048 * 128 * 4
    ia.max_blocks = 16  # short rows: scores only
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_OK
    assert ia.workspace_bytes == 8 * 16 * 128 * 4
    ia.max_blocks = 2048
    ia.topk = 4096
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_INVALID_ARG
    ia.topk = 512
    for heads, want in ((0, b.CSA_ERR_UNSUPPORTED), (1, b.CSA_OK), (32, b.CSA_OK),
                        (128, b.CSA_OK), (129, b.CSA_ERR_UNSUPPORTED)):
        ia.n_heads = heads
        assert L.csa_index_topk(ctypes.byref(ia), None) == want, heads
    ia.head_dim = 64
    ia.n_heads = 64
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_UNSUPPORTED
    ia.head_dim = 128

    # hierarchical indexer: level one adds the block maxima; reindex rows hold
    # n_cand * cand_block candidate entries plus one count per row
    ia.n_heads, ia.max_blocks = 64, 16
    buf = ctypes.create_string_buffer(64)
    ia.cand_block, ia.n_cand, ia.cand_out = 8, 64, ctypes.addressof(buf)
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_OK
    assert ia.workspace_bytes == 8 * 2048 * 4 + 8 * 256 * 4
    ia.cand_out, ia.cand_in = None, ctypes.addressof(buf)
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_OK
    assert ia.workspace_bytes == 8 * 512 * 4 + 256
    ia.cand_block = 12
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_UNSUPPORTED
    ia.cand_block, ia.n_cand = 8, 4096
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_INVALID_ARG
    ia.n_cand, ia.cand_out = 64, ctypes.addressof(buf)  # both modes at once
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_INVALID_ARG
    ia.cand_in = None
    assert L.csa_index_topk_noalloc(ctypes.byref(ia), None) == b.CSA_ERR_UNSUPPORTED
    ia.n_heads = 128  # the hierarchical modes take at most 64 index heads
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_UNSUPPORTED
    ia.n_heads = 64
    # a caller built without the hierarchical fields gets neither mode
    ia.struct_size = b.IndexArgs.cand_block.offset
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_OK
    assert ia.workspace_bytes == 8 * 2048 * 4
    ia.struct_size = b.IndexArgs.cand_block.offset - 8
    assert L.csa_index_topk(ctypes.byref(ia), None) == b.CSA_ERR_INVALID_ARG

    aa = b.AttnArgs()
    aa.struct_size = ctypes.sizeof(aa)
    aa.n_rows, aa.n_heads, aa.head_dim, aa.ratio, aa.topk, aa.window = 8, 64, 512, 4, 2048, 128
    # the decode call merges its split partials through the workspace: per
    # (row, head group) and split 64 KB of partials and 512 bytes of statistics,
    # plus two counters per (row, head group); the split count depends on the
    # device's SM count (one split without a device), at most 17 here
    aa.workspace_bytes = 123
    assert L.csa_sparse_attn_decode(ctypes.byref(aa), None) == b.CSA_OK
    items = 8
    per_split = items * (8 * 512 * 16 + 2 * 64 * 4)
    rest = aa.workspace_bytes - items * 8
    assert rest > 0 and rest % per_split == 0 and 1 <= rest // per_split <= 17
    # the BF16 prefill call keeps its scratch on chip: no workspace
    aa.workspace_bytes = 123
    assert L.csa_sparse_attn_prefill(ctypes.byref(aa), None) == b.CSA_OK
    assert aa.workspace_bytes == 0
    for heads, want in ((0, b.CSA_ERR_UNSUPPORTED), (16, b.CSA_OK), (128, b.CSA_OK),
                        (129, b.CSA_ERR_UNSUPPORTED)):
        aa.n_heads = heads
        assert L.csa_sparse_attn_decode(ctypes.byref(aa), None) == want, heads
        assert L.csa_sparse_attn_prefill(ctypes.byref(aa), None) == want, heads
    aa.n_heads = 64
    aa.window = 64
    assert L.csa_sparse_attn_decode(ctypes.byref(aa), None) == b.CSA_ERR_UNSUPPORTED
