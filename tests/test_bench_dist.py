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


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the float64 oracle on the host (no GPU
    needed) and prints one JSON line with the same metric, unit, direction and
    config keys as the GPU arm."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--cpu-seconds", "1"], capture_output=True, text=True, timeout=600,
                         cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"]
    assert set(line["config"]) == {"workload", "T", "E", "k", "dim", "nfe", "global_batch", "parallelism", "l2",
                                   "timing"}
