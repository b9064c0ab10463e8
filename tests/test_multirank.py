"""The N > 1 path of bench.py on CPU: two gloo ranks (one process each).

bench.py runs one independent replica per GPU under torchrun. Its only
collective is the max over ranks of the step times; the whole-job value is
the bytes all replicas moved divided by that time. The reference arm runs on
rank 0 only. These checks need no GPU.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (1 + r) ms per step and (0.5 + 0.25 r) ms in the kernel
    step_s, kern_s = bench.max_over_ranks([1e-3 * (1 + rank), 1e-3 * (0.5 + 0.25 * rank)], "cpu")
    value = bench.whole_job_gbs(1e9, world, step_s)
    dist.barrier()
    dist.destroy_process_group()
    # the reference arm: only rank 0 does work and prints
    buf = io.StringIO()
    argv = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world)]
    try:
        if rank != 0:
            with redirect_stdout(buf):
                bench.main()
    finally:
        sys.argv = argv
    out.put((rank, step_s, kern_s, value, buf.getvalue()))


def test_two_gloo_ranks_take_the_slowest_replica():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, step_s, kern_s, value, printed in res:
        assert step_s == pytest.approx(2e-3) and kern_s == pytest.approx(0.75e-3)
        # 2 replicas x 1 GB per step in 2 ms = 1000 GB/s
        assert value == pytest.approx(1000.0)
        if rank != 0:
            assert printed == ""  # rank 1 exits without work under torchrun
