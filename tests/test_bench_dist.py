"""The bench's multi-rank aggregation (replicas only) on CPU with gloo, world size 2.

Each rank reports its own units and seconds; the whole-job rate must be the
units of all ranks over the slowest rank's time.
"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist()
    assert d.world == world and d.pg is not None
    d.barrier()
    units, secs = 100.0 * (rank + 1), 0.5 + rank  # rank 1 is slower
    rate, slowest = bench.whole_job_rate(units, secs, d)
    q.put((rank, rate, slowest))
    d.close()


def test_whole_job_rate_over_two_gloo_ranks():
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
    for _, rate, slowest in res:
        assert slowest == 1.5
        assert abs(rate - 300.0 / 1.5) < 1e-9


def test_single_process_is_its_own_world():
    os.environ.pop("WORLD_SIZE", None)
    import bench

    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    assert bench.whole_job_rate(10.0, 2.0, d) == (5.0, 2.0)
