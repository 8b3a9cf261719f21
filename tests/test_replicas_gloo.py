"""The benchmark's multi-GPU mode runs independent replicas (the path does
not shard: its ranks are partitions of one GPU).  Its host-side aggregation -
max time over ranks, whole-job value = all replicas' work / that time - is
checked here with world_size 2 over gloo on CPU."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]
    bench.barrier(world)
    m = bench.reduce_max(local_ms, world)
    v = bench.replica_value(1000.0, 10, m, world)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_two_replicas_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 150.0
        assert v == pytest.approx(2 * 1000.0 * 10 / 0.150)


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.replica_value(10.0, 4, 2000.0, 1) == pytest.approx(20.0)
    b = bench.algorithmic_bytes(4096, 7168, 8, 256, 8, 21688)
    assert b["dispatch"] == 4096 * 7168 * 2 + 4096 * 8 * 12 + 4096 * 8 * 4 + 21688 * (7168 * 2 + 64 + 4)
    assert b["combine"] == 21688 * 7168 * 2 + 4096 * 8 * 4 + 4096 * 7168 * 2
