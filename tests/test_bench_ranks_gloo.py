"""The benchmark's multi-rank aggregation on two gloo ranks (CPU): every rank sees the slowest rank's
time, and the job throughput counts every rank's tokens over that time (weak scaling)."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    import torch.distributed as dist
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=2)
        import bench
        t = bench.max_over_ranks([12.5, 40.0][rank], 2)
        q.put((rank, t, bench.job_throughput(128, 10, 2, t)))
        dist.destroy_process_group()
    except Exception as exc:  # pragma: no cover
        q.put((rank, repr(exc), None))


def test_max_over_ranks_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict((r[0], r[1:]) for r in (q.get(timeout=300) for _ in range(2)))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(2):
        t, v = res[rank]
        assert t == 40.0, t
        assert abs(v - 128 * 10 * 2 / 0.040) < 1e-6
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
