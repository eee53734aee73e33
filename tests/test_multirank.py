"""The benchmark's multi-rank host logic on CPU: two gloo ranks agree on the max-over-ranks time,
pass the barrier, draw distinct per-rank workloads (weak scaling, no data exchange), and only rank 0
runs and prints the reference arm."""
import io
import os
import socket
import sys
import contextlib

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (rank, world, rank)
        t = bench.max_over_ranks(1.5 + rank, world, device="cpu")
        bench.barrier(world)
        w = bench.build_workload(1, bench.rank_seed(1, rank), 64)
        digest = float(np.asarray(w.q_mla, dtype=np.float64).sum() + np.asarray(w.kv_pool, dtype=np.float64).sum())
        # the reference arm: rank 0 alone runs and prints (here: rank != 0 must return with no output)
        printed = ""
        if rank != 0:
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.run_reference(bench.argparse.Namespace(steps=1, warmup=1, config=1, requests=64))
            printed = buf.getvalue()
        out[rank] = (t, digest, printed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 2.5               # max over ranks of 1.5, 2.5
    assert out[0][1] != out[1][1]                      # each rank has its own batch
    assert out[1][2] == ""                             # only rank 0 runs the reference arm
