"""The N > 1 path of bench.py on CPU: two gloo ranks run the same aggregation the GPU job
uses (one independent replica per rank, max over ranks of the timed seconds, whole-job
throughput = all ranks' units over the slowest rank's time).  No GPU is involved."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, _ = bench.dist_env()
        seconds = 1.0 + 0.5 * r                  # rank 1 is the slower one
        rate, slowest = bench.whole_job_rate(1000.0, seconds, w)
        q.put((r, w, rate, slowest, bench.reduce_max(float(10 * r), w)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(2))
    for r, w, rate, slowest, mx in got:
        assert w == 2
        assert slowest == pytest.approx(1.5)           # max over ranks
        assert rate == pytest.approx(2 * 1000.0 / 1.5)  # both ranks' units / slowest time
        assert mx == pytest.approx(10.0)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.whole_job_rate(10.0, 2.0, 1) == (5.0, 2.0)
