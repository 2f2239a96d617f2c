"""The N > 1 path of the benchmark as replicas: two gloo ranks on the CPU
check the max-over-ranks step time, the whole-job rate and that only rank 0
runs the reference arm."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ws, r, _ = bench.dist_info()
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, dist)
    rate = bench.job_throughput(1000.0, ms_max, ws)

    class A:
        workload = bench.ti.LLAMA3_8B_T32K.name
        steps = 1
        warmup = 0

    ref = bench.run_reference(A, r, ws) if r != 0 else "rank0-skipped"
    out[rank] = (ws, r, ms_max, rate, ref)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        ws, r, ms_max, rate, ref = res[rank]
        assert (ws, r) == (world, rank)
        assert ms_max == 15.0  # the slowest rank decides
        assert rate == pytest.approx(2 * 1000.0 / 15e-3)
    assert res[1][4] is None  # only rank 0 times the oracle
