"""The N > 1 host logic of bench.py on CPU: two gloo ranks (replicas only, no collective in
the data path).  Each rank's time is reduced to the slowest rank's; the reference arm runs on
rank 0 alone, the other ranks return without work or output."""
import argparse
import contextlib
import io
import os
import socket

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(10.0 * (rank + 1), torch.device("cpu"))
        out = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(out):
                bench.run_reference(argparse.Namespace(steps=1, warmup=0, gpus=world), rank)
        q.put((rank, slowest, out.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_gate_the_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (v, s) for r, v, s in got}
    assert by_rank[0][0] == by_rank[1][0] == 20.0
    assert by_rank[1][1] == ""


def test_no_process_group_is_a_single_replica():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
