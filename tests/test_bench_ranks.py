"""The bench's multi-replica path on CPU: world_size-2 gloo ranks agree on the
whole-job step time (the slowest rank) and bytes (all ranks)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, total = bench.aggregate_ranks(1.5 + rank, 100.0 * (rank + 1), world)
    q.put((rank, ms, total))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, total in got:
        assert ms == 2.5          # the slower rank's time
        assert total == 300.0     # bytes of both ranks


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(3.0, 7.0, 1) == (3.0, 7.0)
