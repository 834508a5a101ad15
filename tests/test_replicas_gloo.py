"""Host-side logic of multi-GPU replicas on CPU: two gloo ranks, each timing
its own replica; the job's time is the slowest rank's and the value counts
the rows of every rank (no collective on the data path)."""
import os
import sys
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    elapsed = [3.0, 5.0][rank]
    out[rank] = bench.reduce_max(elapsed, ws)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_reduction():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 5.0, 1: 5.0}


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max(2.5, 1) == 2.5


def test_algorithmic_bytes_counts_rejected_q_rows():
    import numpy as np

    import bench
    from speculative_decoding_verification_57_gb300 import workloads as W

    w = W.make_random(name="t", B=4, k=3, V=100, dtype="bf16", seed=1, logit_sigma=1.0, draft_sigma=1.0,
                      temperature=1.0, greedy_rows=1)
    na = np.array([3, 0, 1, 3], np.int32)  # row 0 greedy, rows 1-2 rejected, row 3 bonus
    st = np.zeros(4, np.int32)
    base = 4 * 4 * 100 * 2 + 4 * 3 * 12 + 4 * 12 + 4 * 5 * 4
    assert bench.algorithmic_bytes(w, na, st) == base + 2 * 100 * 4
