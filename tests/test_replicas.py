"""The multi-GPU mode is replicas only: every output of the convolution is independent,
the forward pass has no exchange step, so each rank runs its own copy of the workload and
the job's time is the slowest rank's.  These tests run that host-side logic of bench.py on
two gloo ranks on the CPU (no GPU, no collective on the data path)."""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = 0.010 * (rank + 1)               # rank 1 is the slower replica
    t = bench.max_over_ranks(local, dist, "cpu")
    dist.barrier()
    q.put((rank, local, t, bench.whole_job_rate(1e9, world, t)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_aggregate_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for rank, local, t, rate in results:
        assert t == 0.020                    # every rank sees the max, not its own time
        assert abs(rate - 2 * 1e9 / 0.020) < 1e-3
    assert results[0][1] == 0.010 and results[1][1] == 0.020


def test_single_process_needs_no_collective():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.whole_job_rate(10.0, 1, 0.5) == 20.0
