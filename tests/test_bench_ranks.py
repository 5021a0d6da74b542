"""bench.py's multi-rank aggregation on CPU: two gloo ranks (torchrun's environment variables,
127.0.0.1 rendezvous) meet at the barriers, agree on the slowest rank's timed region, and the
whole-job rate counts every rank's units over that time. One rank without a process group is
the identity."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.ranks_barrier()
    total = bench.max_over_ranks(1.0 + 0.5 * rank, "cpu")  # rank 1 is the slower one
    bench.ranks_barrier()
    q.put((rank, bench.dist_env(), total, bench.whole_job_rate(1024, world, total)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, world, local), total, rate in got:
        assert (r, world, local) == (rank, 2, rank)
        assert total == 1.5
        assert rate == 1024 * 2 / 1.5


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    bench.ranks_barrier()
    assert bench.max_over_ranks(0.25, "cpu") == 0.25
    assert bench.whole_job_rate(1024, 1, 0.5) == 2048
