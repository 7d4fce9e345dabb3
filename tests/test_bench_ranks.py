"""The bench's multi-process logic on CPU with gloo, world size 2: the slowest rank's time is
what every rank reports, and the reference arm runs on rank 0 alone."""
import contextlib
import io
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        args = type("A", (), {"warmup": 0, "steps": 1, "gpus": world})()
        buf = io.StringIO()
        printed = ""
        if rank != 0:                        # rank 0 would time the oracle: not needed here
            with contextlib.redirect_stdout(buf):
                bench.run_reference(args, rank, world)
            printed = buf.getvalue()
        dist.barrier()
        out[rank] = (got, printed)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_reference_rank_zero_only():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == 15.0 and out[1][0] == 15.0
    assert out[1][1] == ""


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
