"""The benchmark's multi-process path on CPU: a world of two gloo ranks.

Decode shards nothing (each rank runs an independent replica), so the only
cross-rank exchange is the bench's own reduction of timings and byte counts
outside the timed region: the slowest rank's time and the sum of the bytes
every replica moved.  The reference arm runs on rank 0 alone.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mx = bench.reduce_over_ranks(1.5 + rank, "max", world)
        sm = bench.reduce_over_ranks(10.0 * (rank + 1), "sum", world)
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_reductions_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # every rank sees the slowest rank's time and the job's total bytes
    assert res == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_alone_the_reduction_is_the_value():
    import bench
    assert bench.reduce_over_ranks(3.25, "max", 1) == 3.25
    assert bench.reduce_over_ranks(7.0, "sum", 1) == 7.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    class Args:
        workload, steps, warmup = "tiny_decode", 1, 3

    assert bench.reference_arm(Args(), 1, 2) is None
    assert capsys.readouterr().out == ""
