"""The multi-rank benchmark logic on CPU with two gloo ranks: every rank
draws its own batch (weak scaling), the job's value is the units of all
ranks over the slowest rank's time, and the barrier / reductions agree."""

import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init("gloo")
    # rank r: 1000*(r+1) units in (r+1)*10 ms
    value, ms_max, units = bench.aggregate(1000.0 * (rank + 1), 10.0 * (rank + 1), dist)
    bench.barrier(dist)
    q.put((rank, value, ms_max, units, bench.rank_seed(1, rank)))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms_max, units, seed in out:
        assert ms_max == 20.0
        assert units == 3000.0
        assert abs(value - 3000.0 / 0.020) < 1e-6
    assert out[0][4] != out[1][4], "ranks must draw different batches"


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE"):
        os.environ.pop(k, None)
    assert bench.dist_init("gloo") is None
    value, ms_max, units = bench.aggregate(500.0, 5.0, None)
    assert (value, ms_max, units) == (100000.0, 5.0, 500.0)
