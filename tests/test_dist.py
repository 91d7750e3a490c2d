"""The N > 1 path of bench.py on CPU: two gloo ranks, each an independent
replica of the workload (no collective on the data path).  Checks the
timing rule (every rank sees the slowest rank's time) and the whole-job
throughput, without a GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [3.0, 5.0][rank]                       # rank 1 is the slower replica
    t = bench.dist_max(local_ms)
    q.put((rank, t, bench.job_gbps(world, 1_000_000_000, t / 10)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_rule_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, gbps in got:
        assert t == 5.0                                # max over ranks
        assert gbps == pytest.approx(2 * 1e9 / 0.5e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench
    assert bench.dist_max(2.5) == 2.5
    assert bench.job_gbps(1, 2_000_000, 1.0) == pytest.approx(2.0)
