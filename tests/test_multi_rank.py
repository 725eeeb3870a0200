"""Multi-rank host logic of bench.py on CPU with the gloo backend.

The hot path shards by independent rows with no data-path collective; the
only cross-rank steps are the barrier around the timed region and the
maximum of the step time over ranks.
"""

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


def _worker(rank, world, port, q):
    import sys
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_env()
    bench.barrier(w)
    m = bench.reduce_max(1.5 + rank * 2.25, w)
    q.put((r, l, w, m))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_reduce_max_and_env_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _, _ in res] == list(range(world))
    assert all(w == world for _, _, w, _ in res)
    assert all(m == 1.5 + (world - 1) * 2.25 for _, _, _, m in res)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
