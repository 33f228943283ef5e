"""Host logic of the multi-rank benchmark on CPU ranks (gloo, world size 2).

Under torchrun every rank runs an independent replica of the workload (batch rows
and channels are independent, so there is no data-path exchange); the job's time is
the slowest rank's and its throughput counts the units of all ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_by_rank, out):
    import torch
    import torch.distributed as dist
    import bench
    from selective_state_space_112_b300.workloads import CONFIGS, make_workload
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(ms_by_rank[rank], dist, torch.device("cpu"))
        value = bench.job_throughput(1000, 10, ms, world)
        # each rank draws its own replica (seed offset by rank), same shapes
        spec = dict(CONFIGS["tiny_f32"])
        spec["seed"] += 1000 * rank
        w = make_workload("tiny_f32", **spec)
        first = float(w.x.reshape(-1)[0])
        firsts = [None] * world
        dist.all_gather_object(firsts, first)
        out.put((rank, ms, value, firsts))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_throughput():
    world, port = 2, _free_port()
    ms_by_rank = [12.5, 20.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms_by_rank, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, firsts in got:
        assert ms == pytest.approx(20.0)  # the slowest rank's time
        assert value == pytest.approx(2 * 1000 * 10 / 0.020)
        assert firsts[0] != firsts[1]  # independent replicas
