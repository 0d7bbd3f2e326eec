"""The N>1 path of bench.py runs independent replicas ("replicas only": the virtual
ranks of a layer live on one GPU); its whole-job figure is all ranks' FLOP over the
slowest rank's time.  Checked with world_size 2 over gloo on the CPU."""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch

    import bench

    def reduce_max(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    ms = [2.0, 4.0][rank]
    value, ms_max = bench.aggregate(1e12, ms, world, reduce_max)
    q.put((rank, value, ms_max))
    dist.destroy_process_group()


def test_replica_aggregation_gloo_world2(repo_root):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree: 2 replicas x 1 TFLOP in the slowest rank's 4 ms = 500 TFLOP/s
    for _, value, ms_max in out:
        assert ms_max == pytest.approx(4.0)
        assert value == pytest.approx(500.0)
