"""The multi-GPU benchmark path runs independent replicas (the layer step does
not shard across GPUs): the whole-job value is the units of all ranks over the
slowest rank's time.  Checked here with two gloo ranks on the CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    seconds = [2.0, 4.0][rank]           # rank 1 is the slowest
    v = bench.job_throughput(seconds, 100, world, device="cpu")
    out[rank] = v
    dist.destroy_process_group()


def test_job_throughput_is_units_over_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 200 / 4.0


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(2.0, 10, 1, device="cpu") == 5.0
