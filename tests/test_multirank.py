"""The N > 1 path of bench.py on the CPU: two ranks as gloo processes.

Each rank is an independent replica (its own seeded rows, no exchange on the data
path); the only collective is the max over ranks of the timed region, and the
reported rate counts every rank's rows over that slowest time.  The reference arm
runs on rank 0 only.
"""
import hashlib
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0, 4.0][rank]  # rank 1 is the slowest
        mx = bench.slowest_rank_ms(ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(64, 10, world, mx)
        w = bench.make_workload("single_stream", rank, 2)
        digest = hashlib.sha256(np.ascontiguousarray(w["target"]).tobytes()).hexdigest()
        ref = bench.run_reference(None, rank) if rank != 0 else "rank0"
        torch.distributed.barrier()
        q.put((rank, mx, rate, digest, ref))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replicas_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == list(range(world))
    assert all(o[1] == 5.0 for o in out)                      # every rank reports the slowest time
    assert all(o[2] == pytest.approx(64 * 10 * world / 5e-3) for o in out)
    assert len({o[3] for o in out}) == world                  # each replica verifies its own rows
    assert all(o[4] is None for o in out if o[0] != 0)        # the reference arm: rank 0 alone


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.slowest_rank_ms(2.5, 1, torch.device("cpu")) == 2.5
    assert bench.whole_job_rate(1, 20000, 1, 140.0) == pytest.approx(20000 / 0.14)
