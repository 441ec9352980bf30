"""Multi-rank path of bench.py on CPU (gloo, world size 2).

The forward does not shard: every (b,h) pair is independent, so N GPUs run N
replicas of the workload.  The only multi-rank logic is the timing reduction
(barrier, then the maximum step time over ranks) and the whole-job throughput
(tokens of all ranks / that maximum).  This test runs that logic in two gloo
processes with different per-rank times."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_env()
    dist = bench.dist_init(w)
    bench.barrier(dist)
    t_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    t_max = bench.max_over_ranks(dist, t_ms)
    tokens_per_rank, steps = 8192, 4
    value = w * tokens_per_rank * steps / (t_max / 1e3)
    q.put((r, w, local, t_max, value))
    dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_value():
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
    for rank, (r, w, local, t_max, value) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert t_max == pytest.approx(20.0)                  # max over ranks
        assert value == pytest.approx(2 * 8192 * 4 / 0.020)  # all ranks' tokens / max time


def test_single_rank_needs_no_process_group(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_init(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
