"""bench.py's multi-rank host logic on two gloo ranks (CPU only).

Under torchrun each rank runs its own seeded batch of the same shape (weak
scaling, no data-path collective), the timed region's device time is the
maximum over ranks, the whole-job rate counts every rank's units, and the
reference arm runs on rank 0 alone.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import make_workload, spec_for


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = spec_for("tiny_decode")
        spec.seed = bench.rank_seed(spec.seed, rank, world)
        wl = make_workload(spec)
        # this rank's device time (ms) for the timed region: rank 1 is slower
        own = 10.0 + 5.0 * rank
        slowest = bench.max_over_ranks(own, dist, "cpu")
        rate = bench.whole_job_rate(spec.n_rows, world, 4, slowest)
        dist.barrier()
        # the reference arm: ranks other than 0 leave without work or output
        ref_rc = bench.main(["--impl", "reference", "--workload", "tiny_decode"]) if rank else None
        out[rank] = (spec.seed, float(wl.t["q"].float().sum()), slowest, rate, ref_rc)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_and_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    (s0, q0, t0, r0, _), (s1, q1, t1, r1, ref1) = res[0], res[1]
    assert s0 != s1 and q0 != q1          # each rank its own batch
    assert t0 == t1 == 15.0               # both report the slowest rank's time
    n_rows = spec_for("tiny_decode").n_rows
    assert r0 == r1 == pytest.approx(n_rows * world * 4 / 0.015)
    assert ref1 == 0                      # rank 1 of the reference arm exits cleanly


def test_single_rank_is_identity():
    assert bench.rank_seed(7, 0, 1) == 7
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(8, 1, 10, 20.0) == pytest.approx(8 * 10 / 0.02)
