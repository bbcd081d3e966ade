"""One CSA step over resident device buffers: main compressor, index-key
compressor, indexer top-k, then sparse attention -- the order the V4 decode
layer calls them ("DeepSeek V4-Flash, MTP point", "Attention paths").

``CsaStep`` owns the outputs and workspaces so that repeated steps allocate
nothing; it is plumbing around the library calls and computes nothing itself.
Both compressors go through one ``csa_compress_pair`` call (one launch for
short chunks), and every call of the step is issued on one stream, where each
kernel is launched as a programmatic dependent of the one before it.
``capture`` records a whole step as a CUDA graph so that a repeated step
costs one launch on the host.

The hierarchical indexer ("DeepSeek V4.1 Flash": a level-one layer selects
candidate blocks of compressed positions; later reindex layers compute their
own index query but select only inside those blocks) is a ``CsaStep`` with
``n_cand`` (level one: it also fills ``cand``) followed by a ``CsaStep`` with
``cand_in`` (reindex: no compressors, the first layer's caches); ``StepChain``
issues such layers back to back as one step.
"""

from __future__ import annotations

import torch

from . import _binding as B


class CsaStep:
    """Buffers and call sequence for one step.

    ``t`` maps names to device tensors: row_req, row_pos, kv_len, n_cmp,
    kv_pool, kv_table, cmp_pool, idx_pool, idx_scale, cmp_table, q, q_idx,
    idx_w, sink, kv_raw, idx_raw, w_gate, ape, w_gate_i, ape_i, rope_cos,
    rope_sin, and optionally the compressors' state rings state_main,
    state_idx with state_table, and the low-bit caches' scale pools kv_scale,
    cmp_scale and idx_kscale (kv_pool MXFP8, cmp_pool FP4 with E4M3 scales,
    idx_pool FP4 with E8M0 scales, all uint8).  ``ratio``, ``topk``, ``prefill`` and
    ``dense`` (HCA) describe the step; ``n_cand`` > 0 makes the indexer also
    select that many candidate blocks of ``cand_block`` positions into
    ``cand`` (level one), and ``cand_in`` restricts it to given candidate
    blocks (reindex).  ``overlap`` makes both compressors pool each entry
    over the previous group's tokens too (the overlapping ratio-4 layout).
    """

    def __init__(self, t: dict, ratio: int, topk: int, prefill: bool = False,
                 compress: bool = True, status: bool = True, dense: bool = False,
                 n_cand: int = 0, cand_block: int = 8, cand_in=None, status_buf=None,
                 overlap: bool = False):
        self.t = t
        self.overlap = bool(overlap)
        self.ratio = int(ratio)
        self.topk = int(topk)
        self.prefill = bool(prefill)
        self.do_compress = bool(compress)
        # HCA: no indexer (and no index-key compressor); the attention takes
        # every visible compressed entry, ``topk`` being the capacity
        self.dense = bool(dense)
        dev = t["q"].device
        T = t["q"].shape[0]
        self.topk_idx = torch.full((T, self.topk), -1, dtype=torch.int32, device=dev)
        self.topk_score = torch.empty((T, self.topk), dtype=torch.float32, device=dev)
        self.out = torch.zeros_like(t["q"])
        self.lse = torch.zeros(t["q"].shape[:2], dtype=torch.float32, device=dev)
        self.status = status_buf if status_buf is not None else (
            torch.zeros(1, dtype=torch.int32, device=dev) if status else None)
        self.cand_block = int(cand_block)
        self.cand = (torch.full((T, int(n_cand)), -1, dtype=torch.int32, device=dev)
                     if n_cand else None)
        self.cand_in = cand_in
        self.lowbit = "cmp_scale" in t
        # low-bit index keys: packed E2M1 (64 bytes a key) or MXFP8 (128 bytes)
        self.key_fmt = ("mxfp8" if self.lowbit and t["idx_pool"].shape[-1] == t["q_idx"].shape[-1]
                        else "fp4")
        # called with the stream right before the attention call (StepIO uses
        # it to wait for the query rows that arrive while the indexer runs)
        self.before_attention = None
        self.ws = {}
        # the indexer's tiling hint (results do not depend on it): rows in pairs
        # unless set to CSA_MODE_PREFILL (rows in fours)
        self.index_mode = B.CSA_MODE_AUTO
        self._prepared = None
        self._graph = None

    def _ws(self, name):
        return self.ws.get(name)

    def _compress_kw(self):
        t = self.t
        main = dict(x=t["kv_raw"], kv=t["kv_raw"], w_gate=t["w_gate"], ape=t["ape"],
                    ratio=self.ratio, positions=t["row_pos"], row_req=t["row_req"],
                    block_table=t["cmp_table"], out="bf16", cmp_pool=t["cmp_pool"],
                    status=self.status)
        keys = dict(x=t["idx_raw"], kv=t["idx_raw"], w_gate=t["w_gate_i"], ape=t["ape_i"],
                    ratio=self.ratio, positions=t["row_pos"], row_req=t["row_req"],
                    block_table=t["cmp_table"], out="int8", idx_pool=t["idx_pool"],
                    idx_scale_pool=t["idx_scale"], rotate=True, rope_cos=t["rope_cos"],
                    rope_sin=t["rope_sin"], status=self.status)
        if self.overlap:
            main.update(overlap=True)
            keys.update(overlap=True)
        if "state_table" in t:  # the compressors' recurrent state rings
            main.update(state_cache=t["state_main"], state_block_table=t["state_table"])
            keys.update(state_cache=t["state_idx"], state_block_table=t["state_table"])
        if self.lowbit:  # publication in the low-bit cache formats
            main.update(out="fp4_e4m3", scale_pool=t["cmp_scale"])
            keys.update(out="mxfp8" if self.key_fmt == "mxfp8" else "fp4_e8m0",
                        cmp_pool=t["idx_pool"], scale_pool=t["idx_kscale"], idx_pool=None,
                        idx_scale_pool=None)
        return main, keys

    def compress(self, stream=None):
        main, keys = self._compress_kw()
        if self.dense:
            self.ws["cm"] = B.csa_compress(workspace=self.ws.get("cm"), stream=stream, **main)
            return
        self.ws["cp"] = B.csa_compress_pair(main, keys, workspaces=self.ws.get("cp", (None, None)),
                                            stream=stream)

    def _index_kw(self):
        t = self.t
        return dict(
            q_idx=t["q_idx"], weights=t["idx_w"], row_req=t["row_req"], row_pos=t["row_pos"],
            n_cmp=t["n_cmp"], ratio=self.ratio, idx_pool=t["idx_pool"],
            idx_scale_pool=t["idx_scale"], cmp_block_table=t["cmp_table"], topk=self.topk,
            topk_idx=self.topk_idx, topk_score=self.topk_score, rope_cos=t["rope_cos"],
            rope_sin=t["rope_sin"],
            mode=self.index_mode, status=self.status,
            cand_out=self.cand, cand_in=self.cand_in, cand_block=self.cand_block,
            key_scale_pool=t.get("idx_kscale"), key_fmt=self.key_fmt)

    def _attn_kw(self):
        t = self.t
        return dict(kv_scale_pool=t.get("kv_scale"), cmp_scale_pool=t.get("cmp_scale"))

    def index(self, stream=None, scores=None):
        self.ws["ix"] = B.csa_index_topk(scores=scores, workspace=self._ws("ix"), stream=stream,
                                         **self._index_kw())

    def _selection(self, topk_idx=None):
        if topk_idx is not None:
            return topk_idx
        return None if self.dense else self.topk_idx

    def attention(self, stream=None, topk_idx=None):
        t = self.t
        fn = B.csa_sparse_attn_prefill if self.prefill else B.csa_sparse_attn_decode
        self.ws["at"] = fn(
            q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], dense_cap=self.topk,
            topk_idx=self._selection(topk_idx), kv_pool=t["kv_pool"],
            kv_block_table=t["kv_table"], kv_len=t["kv_len"], cmp_pool=t["cmp_pool"],
            cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"], ratio=self.ratio, out=self.out,
            lse=self.lse, sink=t["sink"], rope_cos=t["rope_cos"], rope_sin=t["rope_sin"],
            status=self.status, workspace=self._ws("at"), stream=stream, **self._attn_kw())

    def prepare(self):
        """Marshal the step's calls once (buffers must stay in place)."""
        t = self.t
        calls = []
        if self.do_compress:
            main, keys = self._compress_kw()
            calls.append(B.csa_compress(prepare=True, **main) if self.dense else
                         B.csa_compress_pair(main, keys, prepare=True))
        if not self.dense:
            calls.append(B.csa_index_topk(prepare=True, **self._index_kw()))
        fn = B.csa_sparse_attn_prefill if self.prefill else B.csa_sparse_attn_decode
        calls.append(fn(
            q=t["q"], row_req=t["row_req"], row_pos=t["row_pos"], topk_idx=self._selection(),
            dense_cap=self.topk,
            kv_pool=t["kv_pool"], kv_block_table=t["kv_table"], kv_len=t["kv_len"],
            cmp_pool=t["cmp_pool"], cmp_block_table=t["cmp_table"], n_cmp=t["n_cmp"],
            ratio=self.ratio, out=self.out, lse=self.lse, sink=t["sink"],
            rope_cos=t["rope_cos"], rope_sin=t["rope_sin"], status=self.status, prepare=True,
            **self._attn_kw()))
        self._prepared = calls
        return self

    def run(self, stream=None):
        if self._prepared is None:
            if self.do_compress:
                self.compress(stream)
            if not self.dense:
                self.index(stream)
            if self.before_attention:
                self.before_attention(stream)
            self.attention(stream)
        else:
            for i, c in enumerate(self._prepared):
                if i == len(self._prepared) - 1 and self.before_attention:
                    self.before_attention(stream)
                c(stream)
        B.prof_join(stream)

    def capture(self):
        """Record one step (as ``run`` issues it) into a CUDA graph; ``replay``
        then launches the whole step at once.  Call after a warm-up ``run``."""
        if self._prepared is None:
            self.prepare()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.run()
        self._graph = g
        return self

    def replay(self):
        self._graph.replay()

    def drop_graph(self):
        self._graph = None


class StepChain:
    """Layers issued back to back on one stream as one step (e.g. a level-one
    layer and the reindex layer that consumes its candidate blocks)."""

    def __init__(self, steps):
        self.steps = list(steps)
        self._graph = None

    @property
    def status(self):
        return self.steps[0].status

    @property
    def out(self):
        return self.steps[-1].out

    @property
    def lse(self):
        return self.steps[-1].lse

    def prepare(self):
        for s in self.steps:
            s.prepare()
        return self

    def run(self, stream=None):
        for s in self.steps:
            s.run(stream)

    def capture(self):
        for s in self.steps:
            if s._prepared is None:
                s.prepare()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.run()
        self._graph = g
        return self

    def replay(self):
        self._graph.replay()

    def drop_graph(self):
        self._graph = None


class StepIO:
    """A step's per-step inputs packed into one contiguous device block (the
    tensors of ``t`` named in ``names`` become views into it) and its outputs
    into another, each with a pinned host mirror of the same layout: the
    inputs of a step arrive in one host-to-device copy and its outputs leave
    in one device-to-host copy, instead of one copy (and its fixed cost) per
    tensor.  Build it, and bind the outputs, before the step is prepared or
    captured: the step marshals the views' addresses."""

    ALIGN = 256

    def __init__(self, t: dict, names, late=()):
        # inputs only the attention reads (the query rows) go last: they can
        # travel on a side stream while the compressors and the indexer run
        late = [k for k in names if k in set(late)]
        self.names = [k for k in names if k not in set(late)] + late
        self.offsets, off = {}, 0
        for k in self.names:
            if k == (late[0] if late else None):
                self.split = off
            self.offsets[k] = off
            off += self._span(t[k])
        if not late:
            self.split = off
        self._side = None
        self._late_ev = None
        dev = t[self.names[0]].device
        self.dev_in = torch.empty(max(off, 1), dtype=torch.uint8, device=dev)
        self.host_in = torch.empty(max(off, 1), dtype=torch.uint8, pin_memory=True)
        self.in_bytes = 0
        for k in self.names:
            src = t[k]
            nb = src.numel() * src.element_size()
            o = self.offsets[k]
            view = self.dev_in[o:o + nb].view(src.dtype).view(src.shape)
            view.copy_(src)
            self.host_in[o:o + nb].copy_(src.contiguous().view(-1).view(torch.uint8).cpu())
            t[k] = view
            self.in_bytes += nb
        self.dev_out = self.host_out = None
        self.out_bytes = 0

    def _span(self, x):
        nb = x.numel() * x.element_size()
        return (nb + self.ALIGN - 1) // self.ALIGN * self.ALIGN

    def host_input(self, name, like):
        """The pinned host view (dtype and shape of ``like``) where the caller
        writes input ``name`` of the next step."""
        o = self.offsets[name]
        nb = like.numel() * like.element_size()
        return self.host_in[o:o + nb].view(like.dtype).view(like.shape)

    def bind_outputs(self, step):
        """Give ``step`` (a CsaStep, or a StepChain's last layer) out and lse
        tensors that live in one device block with a pinned host mirror."""
        last = step.steps[-1] if isinstance(step, StepChain) else step
        out, lse = last.out, last.lse
        so, sl = self._span(out), self._span(lse)
        self.dev_out = torch.empty(so + sl, dtype=torch.uint8, device=out.device)
        self.host_out = torch.empty(so + sl, dtype=torch.uint8, pin_memory=True)
        nb_o = out.numel() * out.element_size()
        nb_l = lse.numel() * lse.element_size()
        last.out = self.dev_out[:nb_o].view(out.dtype).view(out.shape)
        last.lse = self.dev_out[so:so + nb_l].view(lse.dtype).view(lse.shape)
        self.out_bytes = nb_o + nb_l
        return self

    def h2d(self):
        self.dev_in.copy_(self.host_in, non_blocking=True)

    def _h2d_split(self):
        """The inputs before the split on the current stream; the late ones
        on a side stream, joined by the step right before its attention."""
        main = torch.cuda.current_stream()
        self.dev_in[:self.split].copy_(self.host_in[:self.split], non_blocking=True)
        if self.split >= self.dev_in.numel():
            return
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.dev_in.device)
            self._late_ev = torch.cuda.Event()
        self._side.wait_stream(main)
        with torch.cuda.stream(self._side):
            self.dev_in[self.split:].copy_(self.host_in[self.split:], non_blocking=True)
            self._late_ev.record(self._side)

    def capture(self, step):
        """A CUDA graph of one whole step with its copies: inputs in (the late
        ones overlapping the compressors and the indexer), the step, outputs
        out.  Call after a warm-up ``step.run()``; returns the graph."""
        first = step.steps[0] if isinstance(step, StepChain) else step
        for s_ in (step.steps if isinstance(step, StepChain) else [step]):
            if s_._prepared is None:
                s_.prepare()
        first.before_attention = (lambda stream: torch.cuda.current_stream().wait_event(
            self._late_ev)) if self.split < self.dev_in.numel() else None
        self._h2d_split()  # creates the side stream and event outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self._h2d_split()
            step.run()
            self.d2h()
        return g

    def d2h(self):
        self.host_out.copy_(self.dev_out, non_blocking=True)
