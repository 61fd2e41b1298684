"""The benchmark's multi-GPU path on CPU: two gloo ranks, one independent problem each.

The decode shards into independent problems (one per GPU) with no collective on the data
path; the only exchange is the max over ranks of the time per step.  These tests run the
benchmark's own helpers in two processes on 127.0.0.1.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import shared_prefix_paged_attn_b300 as fa
    dist, r, n, local = bench.dist_setup(world)
    assert (r, n) == (rank, world) and dist is not None
    w = bench.rank_workload(1, rank, "cpu")
    st = fa.plan_for(w).stats()
    ms = 1.0 + rank * 0.25  # a stand-in for this rank's measured time per step
    slowest = bench.max_over_ranks(dist, ms, torch.device("cpu"))
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), q=w.q.float().numpy()[:4],
             unique=st["unique_visible_slots"], seed=w.meta["seed"], slowest=slowest)
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    out = tmp_path_factory.mktemp("ranks")
    mp.start_processes(_rank_main, args=(2, _free_port(), str(out)), nprocs=2, join=True,
                       start_method="spawn")
    return [np.load(out / f"rank{r}.npz") for r in range(2)]


def test_every_rank_gets_the_slowest_time(two_ranks):
    assert [float(d["slowest"]) for d in two_ranks] == [1.25, 1.25]


def test_ranks_solve_independent_problems_of_the_same_shape(two_ranks):
    a, b = two_ranks
    assert int(a["seed"]) != int(b["seed"])
    assert int(a["unique"]) == int(b["unique"])  # same structure, so the same unique KV bytes
    assert not np.array_equal(a["q"], b["q"])    # different values
