"""The N>1 bench path on CPU: two gloo ranks (world size 2) check the
host-side logic bench.py uses under torchrun: every rank gets its own
batch seed (weak scaling, no data-path collective), and the timed figure
is the max over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    seed = bench.shard_seed(7, r)
    slowest = bench.reduce_max(1.5 + r, device="cpu")
    bench.barrier()
    q.put((r, w, seed, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_seed_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == 2 for _, w, _, _ in res)
    assert res[0][2] != res[1][2]             # distinct batches per rank
    assert all(m == 2.5 for *_, m in res)     # max over ranks
