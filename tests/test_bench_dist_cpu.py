"""The benchmark's multi-rank helpers (barrier, max over ranks) on two gloo
ranks on the CPU: every rank must see the slowest rank's time."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world),
                       "GQA_BENCH_BACKEND": "gloo"})
    import bench
    r, w = bench.dist_setup()
    bench.dist_barrier(w)
    results[r] = bench.dist_max(1.5 + r, w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 2.5, 1: 2.5}
