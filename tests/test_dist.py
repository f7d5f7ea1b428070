"""Multi-process host logic of bench.py on the CPU (gloo, world size 2): the
replicas' step times are reduced with a max, and the whole-job value counts
every replica's bytes.  The matvec itself needs no exchange (replicas only)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    local = [1.0 + rank, 10.0 - rank]                     # rank 1 is slower on the first timing
    dev_ms, e2e_ms = bench.max_over_ranks(local, torch.device("cpu"))
    value = bench.aggregate_value(w, 7_973_699_584, dev_ms)
    q.put((r, lr, w, dev_ms, e2e_ms, value))
    dist.destroy_process_group()


def test_replicas_reduce_max_and_sum_bytes():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, lr, w, dev_ms, e2e_ms, value) in enumerate(out):
        assert rank == r and lr == r and w == world
        assert dev_ms == 2.0 and e2e_ms == 10.0            # the slowest replica sets each time
        assert value == pytest.approx(2 * 7_973_699_584 / 2e-3 / 1e9)
