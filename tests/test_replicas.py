"""The multi-GPU path is replicas only: every rank runs the whole forward on its own GPU
and the benchmark reports the max time over ranks.  The host logic of that path (barrier,
max over ranks) runs here as two gloo ranks on the CPU."""
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


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    bench.barrier(ws)
    got = bench.max_over_ranks(1.5 + rank, ws)
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((rank, ws, got))


def test_two_gloo_ranks_report_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2, 2]
    assert all(abs(r[2] - 2.5) < 1e-12 for r in res)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
