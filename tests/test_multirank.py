"""The N>1 host logic of bench.py on CPU: two gloo ranks (world_size 2, replicas only), each
with its own step time; the job's throughput is every rank's tokens over the slowest rank's
time, and both ranks agree on it."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_by_rank, tokens, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    value, ms = bench.job_throughput(ms_by_rank[rank], tokens, world, max_over_ranks)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, value, ms))


def test_two_gloo_ranks_report_the_whole_job_at_the_slowest_pace():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    ms_by_rank = [4.0, 5.0]
    tokens = 32768
    procs = [ctx.Process(target=_rank, args=(r, 2, port, ms_by_rank, tokens, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms in res:
        assert ms == pytest.approx(5.0)
        assert value == pytest.approx(2 * tokens / 5e-3)


def test_one_rank_is_its_own_job():
    value, ms = bench.job_throughput(4.0, 1000, 1, reduce_max=None)
    assert ms == 4.0 and value == pytest.approx(1000 / 4e-3)
