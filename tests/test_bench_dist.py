"""The bench's multi-rank aggregation on two gloo ranks (CPU): whole-job
throughput is the units of all ranks over the slowest rank's time."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, u = bench.aggregate(0.010 * (rank + 1), 4096.0, world)
    out.put((rank, t, u))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in res:
        assert abs(t - 0.020) < 1e-12 and u == 8192.0   # max time, summed tokens


def test_aggregate_single_rank_is_identity():
    import bench
    assert bench.aggregate(0.5, 10.0, 1) == (0.5, 10.0)
