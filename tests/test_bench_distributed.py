"""The bench's multi-rank path on CPU: two gloo ranks, each timing its own
full step (weak scaling), agree on the slowest rank's time, and the job's
throughput counts every rank's bytes over that time."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    ms = bench.max_over_ranks(2.0 + 3.0 * rank, w, "cpu")
    q.put((r, w, lr, ms, bench.job_gbs(10**9, w, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == 5.0 for r in res)                  # max of 2 ms and 5 ms
    assert all(abs(r[4] - 2 * 1e9 / 5e-3 / 1e9) < 1e-9 for r in res)  # 400 GB/s


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_gbs(7 * 10**9, 1, 1.0) == 7000.0
