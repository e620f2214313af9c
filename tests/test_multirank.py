"""The N>1 path of bench.py on CPU: two gloo ranks (replicas only, no data-path
collective) agree on the slowest replica's time and on the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = 100.0 + 50.0 * rank                       # rank 1 is the slow replica
    mx = bench.max_over_ranks(my_ms)
    out[rank] = (mx, bench.job_throughput(4096, 10, world, mx))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    mx, thr = out[0]
    assert mx == 150.0
    assert thr == pytest.approx(4096 * 10 * 2 / 0.150)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(4096, 20, 1, 40.0) == pytest.approx(4096 * 20 / 0.040)
