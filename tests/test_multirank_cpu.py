"""The replica path of the bench on two gloo ranks (CPU): each rank plans its own
copy of the job with the product planner, and the step time is the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import branch_packed_scoring_gb300 as spinf
    from synth import workloads as wl

    inputs = wl.wikinews()
    plan = spinf.Plan(inputs, vocab=262144)
    tokens = sum(plan.pass_info(p).T for p in range(plan.num_passes))
    ms = 1.0 + rank                       # a slower second rank
    slowest = bench.max_over_ranks(ms, world, torch.device("cpu"))
    out[rank] = (tokens, slowest, bench.replica_value(tokens, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas(spinf):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    (t0, s0, v0), (t1, s1, v1) = out[0], out[1]
    assert t0 == t1 == 28616 and s0 == s1 == 2.0
    assert v0 == v1 == pytest.approx(2 * 28616 / 2e-3)
