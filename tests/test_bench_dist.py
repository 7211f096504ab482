"""bench.py's multi-process host logic on CPU: 2 gloo ranks, max-over-ranks timing and the whole-job
value.  No GPU is touched."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        mine = [3.0, 5.5][rank]
        got = bench.reduce_max(mine)
        bench.barrier()
        q.put((rank, got, bench.whole_job_us_per_step(got, w)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [5.5, 5.5]           # both ranks see the slowest rank's time
    assert res[0][2] == pytest.approx(5.5 * 1000 / 2)  # us per layer-step of the whole job


def test_single_process_helpers():
    import bench
    assert bench.reduce_max(2.5) == 2.5
    assert bench.whole_job_us_per_step(1.0, 1) == 1000.0
