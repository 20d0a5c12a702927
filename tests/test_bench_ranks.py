"""The multi-rank bench logic on CPU (gloo, world size 2): the job's step time
is the slowest rank's, and the whole-job value counts every rank's bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [4.0, 5.0][rank]
    m = bench.max_over_ranks(local_ms, world)
    v = bench.weak_scaling_value(1_000_000_000, world, m)
    bench.barrier(world)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, m, v in res:
        assert m == 5.0
        assert v == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_decode_bytes_formula():
    import numpy as np

    import bench
    from workloads import configs
    w = configs.config3()
    b = bench.decode_bytes(w, w.block_tables, w.context_lens)
    # 671 088 640 B of K+V + 655 360 B of q and out + 32*64*4 table entries + 32*4 lengths
    assert b == 671_088_640 + 655_360 + 32 * 64 * 4 + 32 * 4
