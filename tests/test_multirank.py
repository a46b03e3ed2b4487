"""The N > 1 path of bench.py on the CPU: two gloo ranks.

The path does not shard within a chunk (replicas only): every rank denoises its
own chunks and the job's time is the slowest rank's.  These tests run the
aggregation bench.py uses, with a gloo all-reduce in place of NCCL, and the
reference arm's rank rule (rank 0 alone works and prints).
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, steps, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        def reduce_max(v):
            t = torch.tensor([v], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())

        r, _, w = bench.dist_info()
        ms_step, ms_chunk = bench.job_ms_per_chunk(elapsed[rank], steps, w, reduce_max)
        # the reference arm: only rank 0 does work and prints
        buf = io.StringIO()
        args = type("A", (), {"steps": 0, "warmup": 0, "gpus": w})()
        if r != 0:
            with redirect_stdout(buf):
                bench.run_reference(args)
        dist.barrier()
        out.put((r, w, ms_step, ms_chunk, buf.getvalue()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("elapsed", [(10.0, 12.5), (30.0, 7.0)])
def test_replicas_take_the_slowest_rank(elapsed):
    world, steps = 2, 5
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, elapsed, steps, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    t_max = max(elapsed)
    for r, w, ms_step, ms_chunk, printed in res:
        assert w == world
        assert ms_step == pytest.approx(t_max / steps)
        assert ms_chunk == pytest.approx(t_max / (steps * world))   # whole-job time per chunk
        if r != 0:
            assert printed == ""                                     # rank != 0 exits without work
