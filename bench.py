"""Benchmark of the CSA hot path on GB300.

One step = one pass of the whole path over one batch: the main compressor,
the index-key compressor, the indexer top-k and the sparse attention (decode
or prefill).  Default workload: million-position decode (4 requests x 2
rows, contexts of 1,048,576 positions, ratio 4, top-k 2048), the largest
single-GPU configuration.  Other workloads: --workload tiny_decode |
serving_decode | ratio1_decode | chunked_prefill | stateful_decode |
hca_decode | hca_prefill | hier_decode (a level-one layer and a reindex layer
of the hierarchical indexer as one step) | lowbit_decode | lowbit_million (the
low-bit cache formats).

The step is timed as one CUDA graph per step (the headline ``value``) and,
beside it, issued eagerly call by call (``eager``).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a bounded sample of the same workload).
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA decode token-rows/s + % HBM roofline; prefill tokens/s + % tensor roofline"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2

# DRAM traffic per launch from an ncu capture, keyed by kernel; each entry
# names the source it was taken on (sha1 of the kernel's .cu) so a changed
# kernel reports null.  Values are from `ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum` captures of these same bench workloads.
NCU_TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch (one-kernel ncu
    # captures, profiles/dram_traffic.md), keyed by the hash of the kernel's
    # source and the shared headers
    ("tiny_decode", "attn_decode"): {"bytes": 557310, "src": "3c516bde6e00"},
    ("tiny_decode", "index_score"): {"bytes": 168448, "src": "5a17c226935a"},
    ("serving_decode", "attn_decode"): {"bytes": 4609280, "src": "3c516bde6e00"},
    ("serving_decode", "index_score"): {"bytes": 1558784, "src": "5a17c226935a"},
    ("ratio1_decode", "index_score"): {"bytes": 70123776, "src": "5a17c226935a"},
    ("ratio1_decode", "index_topk"): {"bytes": 4454144, "src": "4a72031579c9"},
    ("million_decode", "index_score"): {"bytes": 142287616, "src": "5a17c226935a"},
    ("million_decode", "attn_decode"): {"bytes": 17844736, "src": "3c516bde6e00"},
    ("million_decode", "index_topk"): {"bytes": 8648704, "src": "4a72031579c9"},
    ("chunked_prefill", "attn_prefill"): {"bytes": 1061745408, "src": "6c2a1d534303"},
    ("chunked_prefill", "index_score"): {"bytes": 151614976, "src": "5a17c226935a"},
}


def _env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ---------------------------------------------------------------- multi-rank host logic


def rank_seed(seed, rank, world):
    """Weak scaling: every rank runs its own batch of the same shape."""
    return seed + 1000 * rank if world > 1 else seed


def max_over_ranks(x, dist=None, device="cpu"):
    """The slowest rank's time (identity on one rank)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, steps, total_ms):
    """Units every rank processed, per second of the slowest rank's time."""
    return units_per_rank * world * steps / (total_ms / 1e3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------- algorithmic work


def algorithmic_work(wl):
    """Per-kernel algorithmic bytes and FLOPs of one step: each distinct byte
    a kernel must read or write once, from the workload's shapes only."""
    s = wl.spec
    T = s.n_rows
    rows = [(int(wl.row_req[i]), int(wl.row_pos[i])) for i in range(T)]
    rows = [(b, p) for b, p in rows if b >= 0]
    n_cmp = [int(x) for x in wl.n_cmp]
    vis = [max(0, min(n_cmp[b], (p + 1) // s.ratio)) for b, p in rows]
    req_vis = {}
    for (b, _), v in zip(rows, vis):
        req_vis[b] = max(req_vis.get(b, 0), v)
    H, D, Hi, Di, W = s.heads, s.head_dim, s.idx_heads, s.idx_dim, s.window
    sel = [min(s.topk, v) for v in vis]
    win = [min(W, p + 1) for _, p in rows]
    # bytes of one cached row: index key, compressed KV row, window KV row
    # (low-bit caches: FP4 codes + scale bytes, MXFP8 codes + scale bytes)
    key_b = Di // 2 + Di // 32 if s.lowbit else Di + 4
    cmp_b = D // 2 + D // 16 if s.lowbit else D * 2
    win_b = D + D // 32 if s.lowbit else D * 2
    idx_bytes = sum(v * key_b for v in req_vis.values()) + len(rows) * Hi * (Di * 2 + 4)
    idx_flops = sum(2 * Hi * Di * v for v in vis)
    if s.mode == "prefill":
        # window rows are shared by neighbouring query rows: count each once
        attn_bytes = (len(rows) * H * D * 2 * 2 + sum(n_cmp) * cmp_b +
                      sum(int(x) for x in wl.kv_len) * win_b)
    else:
        attn_bytes = (sum(sel) * cmp_b + len(req_vis) * (W + 1) * win_b +
                      len(rows) * H * D * 2 * 2 + sum(sel) * 4)
    attn_flops = sum(4 * H * D * (k + w) for k, w in zip(sel, win))
    topk_bytes = sum(vis) * 4 + len(rows) * s.topk * 8
    if s.n_cand:
        # hierarchical indexer: the level-one layer also writes each row's block
        # maxima and selects n_cand blocks; the reindex layer reads each row's
        # candidate keys (Vc entries), selects among them and attends again
        cb = s.cand_block
        nblk = [(v + cb - 1) // cb for v in vis]
        vc = [min(v, s.n_cand * cb) for v in vis]
        sel2 = [min(s.topk, v) for v in vc]
        idx_bytes += (sum(nblk) * 4 + sum(v * key_b for v in vc) +
                      len(rows) * (Hi * (Di * 2 + 4) + s.n_cand * 4))
        idx_flops += sum(2 * Hi * Di * v for v in vc)
        topk_bytes += (sum(nblk) * 4 + len(rows) * s.n_cand * 4 +
                       sum(vc) * 4 + len(rows) * s.topk * 8)
        attn_bytes += (sum(sel2) * cmp_b + len(req_vis) * (W + 1) * win_b +
                       len(rows) * H * D * 2 * 2 + sum(sel2) * 4)
        attn_flops += sum(4 * H * D * (k + w) for k, w in zip(sel2, win))
    # compressors (main: x, kv [T, D] BF16 -> BF16 rows; index keys: [T, Di] ->
    # INT8 rows + FP32 scale); a group is r consecutive rows of one request
    # ending at a position p with p % r == r - 1
    r = s.ratio
    rr, rp = [int(x) for x in wl.row_req], [int(x) for x in wl.row_pos]
    def in_chunk(i, j):  # row i - j is the same request at position p_i - j
        return i - j >= 0 and rr[i - j] == rr[i] and rp[i - j] == rp[i] - j
    closing = [i for i in range(T) if rr[i] >= 0 and rp[i] >= 0 and rp[i] % r == r - 1]
    # tokens a closing row pools: its group, or with overlap the previous group too
    span = {i: min(rp[i] + 1, 2 * r) if s.overlap else r for i in closing}
    if s.state:
        # with state rings every closing row publishes; predecessors before the
        # chunk come from the ring and the last `cap` rows of each request write it
        cap = max(4, r) * (2 if s.overlap else 1)
        groups = len(closing)
        ring_reads = sum(1 for i in closing for j in range(1, span[i]) if not in_chunk(i, j))
        ring_writes = sum(1 for i in range(T) if rr[i] >= 0 and rp[i] >= 0 and
                          not (i + cap < T and rr[i + cap] == rr[i]))
    else:
        groups = sum(1 for i in closing if all(in_chunk(i, j) for j in range(1, span[i])))
        ring_reads = ring_writes = 0
    # (d, output bytes per group); HCA (dense) runs only the main compressor
    dims = ((D, cmp_b),) if s.dense else ((D, cmp_b), (Di, key_b))
    w_bytes = sum(d * d * 2 + r * d * 4 for d, _ in dims)    # W_gate and ape
    out_bytes = sum(groups * ob for _, ob in dims)
    ring_bytes = sum((ring_reads + ring_writes) * 2 * d * 4 for d, _ in dims)
    gate_flops = sum(2 * T * d * d for d, _ in dims)
    return {
        "index_score": {"bytes": idx_bytes, "flops": idx_flops},
        "index_topk": {"bytes": topk_bytes, "flops": 0},
        "attn_decode": {"bytes": attn_bytes, "flops": attn_flops},
        "attn_prefill": {"bytes": attn_bytes, "flops": attn_flops},
        # long chunks: x and W_gate in, FP32 logits out; then logits and kv in, rows out
        "compress_gate": {"bytes": w_bytes + sum(T * d * (2 + 4) for d, _ in dims),
                          "flops": gate_flops},
        "compress_pool": {"bytes": sum(T * d * (4 + 2) for d, _ in dims) + out_bytes +
                          ring_bytes, "flops": 0},
        # short chunks: W_gate, ape and the r rows of x and kv of every group in, rows out
        "compress_fused": {"bytes": w_bytes + sum(groups * r * d * 2 * 2 for d, _ in dims) +
                           out_bytes, "flops": sum(2 * groups * r * d * d for d, _ in dims)},
        # low-bit prefill: every mapped page of both pools read once, written as BF16
        "dequant": {"bytes": (sum(n_cmp) * (cmp_b + D * 2) +
                              sum(int(x) for x in wl.kv_len) * (win_b + D * 2)), "flops": 0},
        "_rows": len(rows),
    }


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples (every 20 ms) taken during the timed region, which
    ``mark_start``/``mark_end`` delimit; a region shorter than one sampling
    period reports the sample nearest to it."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 3.0
            while not self.lines and time.time() < deadline:  # sampling is running
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(0.05)  # the first sample after the region, for short regions

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = list(self.lines)
        window = "timed region"
        if self.t0 is not None and self.t1 is not None:
            inside = [ln for t, ln in lines if self.t0 <= t <= self.t1]
            if not inside:
                after = [ln for t, ln in lines if t > self.t1]
                inside = after[:1]
                window = "first sample after the timed region (region shorter than 20 ms)"
            lines = inside
        else:
            lines = [ln for _, ln in lines]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


# ---------------------------------------------------------------- reference arm (CPU oracle)


def _oracle_threads():
    """Threads the oracle uses: its row loop runs in one Python thread, and
    numpy's BLAS (matrix products) runs on the BLAS thread pool.  Returns
    (threads, description)."""
    blas = None
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            blas = int(max(n))
    except Exception:  # threadpoolctl is optional
        pass
    if blas is None:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                blas = int(os.environ[var])
                break
    if blas is None:
        blas = os.cpu_count() or 1
    desc = (f"one Python thread drives the oracle's per-row loop; numpy's BLAS calls "
            f"use up to {blas} threads; the host has {os.cpu_count()} cores")
    return blas, desc


def _cpu_line(rate, unit, desc):
    threads, how = _oracle_threads()
    return {"value": rate, "unit": unit, "cores": threads, "nproc": os.cpu_count(),
            "threads": how, "kind": "oracle", "sample": desc}


def oracle_sample(wl, budget_s=10.0, max_rows=None):
    """Time the oracle's chain (compress, scores, top-k, attention) on a bounded
    sample of the workload: whole passes over the step's rows (the
    compression of the chunk, then every row) repeated until ``budget_s`` has
    passed, or, when one pass takes longer, the rows of the first pass done
    by then with the compression charged per row in proportion.  Returns
    (rows/s, description, rows done)."""
    from oracle import select_blocks, topk_in_blocks, topk_select
    from oracle import step as OS

    s = wl.spec
    rows = [i for i in range(s.n_rows) if int(wl.row_req[i]) >= 0]
    if max_rows is not None:
        rows = rows[:max_rows]
    t2 = OS.reindex_tensors(wl.t) if s.n_cand else None
    t_start = time.perf_counter()
    done = passes = 0
    t_comp = t_rows = 0.0
    while True:
        t0 = time.perf_counter()
        pools, _, _ = OS.compress_step(wl.t, s)
        t1 = time.perf_counter()
        t_comp += t1 - t0
        n = 0
        for row in rows:
            sc = OS.index_row(wl.t, s, pools, row)
            sel = topk_select(sc, s.topk)
            OS.attention_row(wl.t, s, pools, row, sel)
            if s.n_cand:  # level-one blocks, then the reindex layer
                cand = select_blocks(sc, s.n_cand, s.cand_block)
                sc2 = OS.index_row(t2, s, pools, row)
                OS.attention_row(t2, s, pools, row,
                                 topk_in_blocks(sc2, cand, s.topk, s.cand_block))
            n += 1
            if time.perf_counter() - t_start > budget_s:
                break
        t_rows += time.perf_counter() - t1
        done += n
        if n == len(rows):
            passes += 1
        if time.perf_counter() - t_start > budget_s or n < len(rows):
            break
    if passes:
        rate = passes * len(rows) / (time.perf_counter() - t_start)
        desc = (f"oracle chain (compression of the chunk, then scores, top-k and attention "
                f"per row) over the {len(rows)} rows of {s.name}, repeated: {passes} whole "
                f"passes in {time.perf_counter() - t_start:.1f}s")
        return rate, desc, passes * len(rows)
    per_row = t_rows / max(1, done) + t_comp / max(1, len(rows))
    desc = (f"oracle chain on {done} of {len(rows)} rows of {s.name} "
            f"(compression of the whole chunk {t_comp:.2f}s, rows {t_rows:.2f}s)")
    return 1.0 / per_row, desc, done


def run_reference(args, wl):
    rate, desc, done = oracle_sample(wl, budget_s=args.ref_budget)
    unit = "tokens/s" if wl.spec.mode == "prefill" else "token_rows/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(wl, args),
        "cpu_baseline": _cpu_line(rate, unit, desc),
        "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(wl, args):
    s = wl.spec
    c = {"workload": s.name, "requests": s.n_req, "rows": s.n_rows, "contexts": s.ctx,
         "ratio": s.ratio, "topk": s.topk, "heads": s.heads, "head_dim": s.head_dim,
         "idx_heads": s.idx_heads, "idx_dim": s.idx_dim, "window": s.window,
         "l2": "flushed before every timed step (256 MiB write)",
         "parallelism": f"replicas x{args.gpus}"}
    if s.n_cand:
        c.update(layers=["level-one", "reindex"], n_cand=s.n_cand, cand_block=s.cand_block)
    if s.lowbit:
        c.update(caches={"window": "MXFP8 (E4M3, E8M0 per 32)",
                         "compressed": "FP4 (E2M1, E4M3 per 16)",
                         "index_keys": "FP4 (E2M1, E8M0 per 32)"})
    return c


# ---------------------------------------------------------------- GPU arm


def _src_sha(name):
    """Hash of a kernel's source file and of every shared header it may
    include: a stored traffic figure counts only while both are unchanged."""
    csrc = os.path.join(ROOT, "prefill_csa_compress_gb300", "csrc")
    h = hashlib.sha1()
    try:
        for path in [os.path.join(csrc, name)] + sorted(glob.glob(os.path.join(csrc, "*.cuh"))):
            h.update(open(path, "rb").read())
    except OSError:
        return None
    return h.hexdigest()[:12]


KERNEL_SRC = {"index_score": "k_index_tc.cu", "index_topk": "k_index.cu",
              "attn_decode": "k_attn.cu", "attn_prefill": "k_attn_prefill.cu",
              "compress_gate": "k_compress.cu", "compress_pool": "k_compress.cu",
              "compress_fused": "k_compress.cu", "dequant": "k_dequant.cu"}


def run_gpu(args, wl, rank, world, local_rank):
    import torch

    import prefill_csa_compress_gb300 as csa
    from prefill_csa_compress_gb300.pipeline import CsaStep

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    s = wl.spec
    t = wl.to(dev)
    prefill = s.mode == "prefill"

    def make_step(t, io=None):
        if s.n_cand:
            # hierarchical indexer: a level-one layer, then a reindex layer over
            # the same caches with its own activations
            from prefill_csa_compress_gb300.pipeline import StepChain
            from workloads import reindex_view

            s1 = CsaStep(t, s.ratio, s.topk, prefill=prefill, n_cand=s.n_cand,
                         cand_block=s.cand_block, overlap=s.overlap)
            s2 = CsaStep(reindex_view(t), s.ratio, s.topk, prefill=prefill, compress=False,
                         cand_in=s1.cand, cand_block=s.cand_block, status_buf=s1.status)
            st = StepChain([s1, s2])
        else:
            st = CsaStep(t, s.ratio, s.topk, prefill=prefill, dense=s.dense, overlap=s.overlap)
        if io is not None:
            io.bind_outputs(st)
        return st.prepare()

    step = make_step(t)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    work = algorithmic_work(wl)
    units = work["_rows"]

    def flush_l2():
        flush.fill_(1)

    # ---- warm-up (also finds the dominant kernel)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    kernels = ["index_score", "index_topk", "attn_prefill" if prefill else "attn_decode",
               "compress_gate", "compress_pool", "compress_fused"]
    if s.lowbit and prefill:
        kernels.append("dequant")
    # per-kernel durations: the step captured with that kernel's event pairs,
    # its calls issued one after another on one stream (no kernel shares the
    # GPU with the timed one), replayed three times with L2 flushed before each
    per_kernel = {}
    for k in kernels:
        csa.prof_enable(k, 16)
        step.capture()
        tot, cnt = 0.0, 0
        for _ in range(3):
            flush_l2()
            step.replay()
            torch.cuda.synchronize()
            ms, n = csa.prof_read(k)
            tot += ms
            cnt += n
        step.drop_graph()
        csa.prof_disable()
        if cnt:
            per_kernel[k] = {"ms_per_launch": tot / cnt, "launches_per_step": cnt / 3}
    dominant = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_launch"] *
                   per_kernel[k]["launches_per_step"])
    launches_per_step = None

    # ---- the step as one CUDA graph (one host launch per step, so the device
    # never waits for the host); the dominant kernel's event pair is recorded
    # inside the graph, so its duration is read back after every replay
    csa.prof_enable(dominant, 16)
    lc0 = csa.launch_count()
    step.capture()
    launches_per_step = csa.launch_count() - lc0
    step.replay()
    torch.cuda.synchronize()

    # ---- timed region: device time of exactly K steps, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    dom_ms, dom_n = 0.0, 0
    wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clk:
        clk.mark_start()
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            step.replay()
            ev[i][1].record(stream)
            ev[i][1].synchronize()
            ms, n = csa.prof_read(dominant)
            dom_ms += ms
            dom_n += n
        torch.cuda.synchronize()
        clk.mark_end()
    wall = time.perf_counter() - wall0
    launches = launches_per_step * args.steps
    if dist:
        dist.barrier()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dist, dev)

    # ---- the same K steps issued eagerly (the step's calls one by one from
    # the host, each crossing the C ABI), L2 flushed before each
    step.drop_graph()
    csa.prof_disable()
    ev_e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()
        ev_e[i][0].record(stream)
        step.run()
        ev_e[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev_e), dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(units, world, args.steps, total_ms)
    status = int(step.status.item())

    # ---- end to end through the public API with host buffers: the step's
    # per-step inputs packed into one pinned host block and one device block
    # (one host-to-device copy per step), out and lse likewise (one copy
    # back), around the step's graph
    from prefill_csa_compress_gb300.pipeline import StepIO

    per_step_inputs = ["q", "q_idx", "idx_w", "kv_raw", "idx_raw", "row_req", "row_pos",
                       "kv_len", "n_cmp"]
    if s.n_cand:
        per_step_inputs += ["q2", "q_idx2", "idx_w2"]
    t_e = dict(t)
    io = StepIO(t_e, per_step_inputs)
    step_e = make_step(t_e, io)
    step_e.run()
    torch.cuda.synchronize()
    step_e.capture()
    bi, bo = io.in_bytes, io.out_bytes
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()
        ee[i][0].record(stream)
        io.h2d()
        step_e.replay()
        io.d2h()
        ee[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ee), dist, dev)
    e2e_value = whole_job_rate(units, world, args.steps, e2e_ms)
    step_e.drop_graph()

    # ---- roofline of the dominant kernel
    peaks = _peaks()
    dom_avg_ms = dom_ms / max(1, dom_n)
    w = work[dominant]
    n_per_step = max(1.0, per_kernel[dominant]["launches_per_step"])
    if prefill and w["flops"] > 0 and dominant in ("attn_prefill", "index_score", "compress_gate"):
        achieved = w["flops"] / n_per_step / (dom_avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"]}
    else:
        per_launch = w["bytes"] / n_per_step
        achieved = per_launch / (dom_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    tr = NCU_TRAFFIC.get((s.name, dominant))
    roof["traffic"] = tr["bytes"] if tr and tr["src"] == _src_sha(KERNEL_SRC[dominant]) else None
    roof["kernel"] = dominant
    roof["kernel_ms"] = dom_avg_ms
    roof["peak_source"] = peaks["source"]

    result = None
    if rank == 0:
        unit = "tokens/s" if prefill else "token_rows/s"
        result = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": _config(wl, args), "roofline": roof,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo},
            "eager": {"value": whole_job_rate(units, world, args.steps, eager_ms), "unit": unit,
                      "ms_per_step": eager_ms / args.steps,
                      "how": "the step's calls issued one by one through the C ABI, no graph"},
            "gpu_launches": launches, "launches_per_step": launches_per_step,
            "clocks": clk.summary(), "wall_s": wall, "device_status": status,
            "per_kernel_ms": {k: v["ms_per_launch"] * v["launches_per_step"]
                              for k, v in per_kernel.items()},
        }
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="million_decode")
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = _env_rank()

    from workloads import make_workload, spec_for

    if args.impl == "reference":
        if rank != 0:
            return 0
        run_reference(args, make_workload(spec_for(args.workload)))
        return 0

    spec = spec_for(args.workload)
    spec.seed = rank_seed(spec.seed, rank, world)
    wl = make_workload(spec)
    # the oracle's CPU timing runs before any CUDA work (no fork after CUDA init)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc, _ = oracle_sample(wl, budget_s=args.ref_budget)
        cpu = _cpu_line(rate, "tokens/s" if spec.mode == "prefill" else "token_rows/s", desc)
    res = run_gpu(args, wl, rank, world, local_rank)
    if rank == 0:
        res["cpu_baseline"] = cpu
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
