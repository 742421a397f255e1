"""bench.py's multi-GPU path is replicas only: each rank times its own batch,
the step time is the maximum over ranks and the job throughput counts every
rank's tokens.  Checked with two gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    bench.barrier(world)
    my_ms = [2.5, 3.0][rank]
    ms = bench.max_over_ranks(my_ms, world, device="cpu")
    out[rank] = (ms, bench.job_tokens_per_s(4112, world, ms))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.0
    assert abs(res[0][1] - 2 * 4112 / 3.0e-3) < 1e-6
