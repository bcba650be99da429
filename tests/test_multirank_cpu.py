"""The benchmark's multi-rank control path on CPU: two gloo ranks launched the
way torchrun would (RANK / WORLD_SIZE / MASTER_ADDR=127.0.0.1), each reporting
its own timing; the job's time is the slowest rank's and the throughput counts
every rank's work (replicas, weak scaling).  No GPU and no data-path
collective is involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_info()
    dist.init_process_group("gloo")
    dist.barrier()
    own = [1.0 + r, 10.0 - 3 * r, 0.5 * (r + 1)]
    got = bench.max_over_ranks(dist, own)
    value = bench.throughput(w, 5, 1000, got[0])
    dist.destroy_process_group()
    q.put((r, w, local, got, value))


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, got, value) in enumerate(results):
        assert (rank, world, local) == (r, 2, r)
        assert got == [2.0, 10.0, 1.0]
        assert value == pytest.approx(2 * 5 * 1000 / 2.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(None, [3, 4.5]) == [3.0, 4.5]
    assert bench.throughput(1, 2, 10, 4.0) == 5.0
