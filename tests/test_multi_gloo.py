"""The multi-GPU path is replicas only: each rank decodes its own sessions and the
only cross-rank steps are bench.py's barrier and max-over-ranks of the timed region.
Exercise those with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    bench.barrier(ws)
    t = bench.max_over_ranks(1.5 + rank, ws)        # per-rank seconds
    value = ws * 4 * 10 / t                          # B=4 sessions, 10 frames per rank
    q.put((r, local, ws, t, value))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and [r[1] for r in res] == [0, 1]
    assert all(r[2] == 2 for r in res)
    assert all(r[3] == 2.5 for r in res)            # the slowest rank's time
    assert all(abs(r[4] - 2 * 4 * 10 / 2.5) < 1e-9 for r in res)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
