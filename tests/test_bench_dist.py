"""bench.py's multi-rank plumbing (one process per GPU under torch.distributed.run)
with world_size 2 on the gloo backend, on the CPU: rank setup, the timing barrier,
the max over ranks of a per-rank time, and the reference arm doing its work on
rank 0 only.  No GPU and no layer call is involved."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    b = _load_bench()
    r, ws, dist = b.dist_setup(world)
    assert (r, ws) == (rank, world) and dist is not None
    b.barrier(dist)
    slowest = b.max_over_ranks(1.5 + rank, dist)   # per-rank ms per step
    # the reference arm: only rank 0 works and reports, the others return nothing
    ref = b.run_reference(None, r, ws) if r != 0 else "rank0"
    dist.destroy_process_group()
    out[rank] = (slowest, ref)


def test_two_rank_barrier_max_and_reference_arm():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == pytest.approx(2.5) and out[1][0] == pytest.approx(2.5)
    assert out[1][1] is None
