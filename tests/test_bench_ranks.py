"""The replica path of bench.py on the CPU: two gloo ranks agree on the slowest rank's time and on the whole-job
figure, as the N-GPU run does over NCCL (replicas only: the decode path has no exchange step)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", init_method="env://")
    try:
        w, r, lr = bench.ranks_from_env()
        dist.barrier()
        slowest = bench.max_over_ranks(times[r], w, "cpu")
        out.put((r, w, lr, slowest, bench.whole_job_gbps(w, 1_000_000, 10, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [3.0, 5.5]   # ms over 10 steps per rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, w, lr, slowest, gbps) in enumerate(res):
        assert (rank, w, lr) == (r, world, r)
        assert slowest == max(times)
        # 2 replicas x 1 MB x 10 steps in 5.5 ms
        assert gbps == pytest.approx(2 * 1_000_000 * 10 / 5.5e-3 / 1e9)


def test_single_rank_is_unchanged():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.whole_job_gbps(1, 37_748_736, 100, 2.2) == pytest.approx(37_748_736 * 100 / 2.2e-3 / 1e9)
