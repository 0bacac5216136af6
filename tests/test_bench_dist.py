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


def _share_rank(rank, port, out):
    import hashlib
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    import synth
    cfg = synth.DIT.with_(n_segments=3, tokens=8, hidden=64, ffn=128)
    hs = bench.shared_host_stack(cfg, rank, dist.barrier)
    digest = hashlib.sha256(hs.buffer.tobytes()).hexdigest()
    views = hashlib.sha256(hs.seg_views[2][2].tobytes()).hexdigest()
    dist.barrier()                       # both have read before either unmaps
    hs.close()
    out.put((rank, digest, views))
    dist.destroy_process_group()


def test_ranks_of_a_node_can_share_one_host_stack():
    """When N copies of the stack do not fit the host, the bench's ranks on a node map one
    stack drawn by local rank 0: the other rank sees exactly the bytes a private draw has."""
    import hashlib
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_share_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (d, v)) for r, d, v in (q.get(timeout=120) for _ in range(2)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg = synth.DIT.with_(n_segments=3, tokens=8, hidden=64, ffn=128)
    ref = synth.HostStack(cfg)
    assert res[0] == res[1]
    assert res[1][0] == hashlib.sha256(ref.buffer.tobytes()).hexdigest()
    assert res[1][1] == hashlib.sha256(ref.seg_views[2][2].tobytes()).hexdigest()
