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


def _split_main(rank, world, port, out_dir):
    # one problem split over the ranks (by KV head, then by request); each rank runs the
    # oracle on its share and rank 0 puts the shares back together
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    dist.init_process_group("gloo")
    w = W.make(5, small=True)
    threads = max(1, oracle.threads_default() // world)
    res = {}
    sub = shard.split_by_kv_head(w, rank, world)
    o, l = oracle.fork_attn(sub, threads=threads)
    got = [None] * world
    dist.all_gather_object(got, (o.reshape(sub.total_q, sub.num_q_heads, -1),
                                 l.reshape(sub.total_q, sub.num_q_heads)))
    res["head"] = got
    sub, mine = shard.split_by_request(w, rank, world)
    o, l = oracle.fork_attn(sub, threads=threads)
    got = [None] * world
    dist.all_gather_object(got, (mine, o.reshape(sub.total_q, sub.num_q_heads, -1),
                                 l.reshape(sub.total_q, sub.num_q_heads),
                                 oracle.unique_slots(sub)[0]))
    res["request"] = got
    if rank == 0:
        import pickle
        with open(os.path.join(out_dir, "split.pkl"), "wb") as f:
            pickle.dump(res, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def split_ranks(tmp_path_factory):
    out = tmp_path_factory.mktemp("split")
    mp.start_processes(_split_main, args=(2, _free_port(), str(out)), nprocs=2, join=True,
                       start_method="spawn")
    import pickle
    with open(out / "split.pkl", "rb") as f:
        return pickle.load(f)


def test_split_by_kv_head_concatenates_to_the_whole_problem_bitwise(split_ranks):
    import oracle
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    w = W.make(5, small=True)
    ref_o, ref_l = oracle.fork_attn(w)
    parts = split_ranks["head"]
    assert [p[1].shape[1] for p in parts] == [16, 16]
    o = shard.gather_heads([torch.from_numpy(p[0]) for p in parts], w).numpy()
    l = shard.gather_heads([torch.from_numpy(p[1]) for p in parts], w).numpy()
    assert np.array_equal(o.reshape(-1, 128), ref_o) and np.array_equal(l.reshape(-1), ref_l)


def test_split_by_request_concatenates_to_the_whole_problem_bitwise(split_ranks):
    import oracle
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    w = W.make(5, small=True)
    ref_o, ref_l = oracle.fork_attn(w)
    parts = split_ranks["request"]
    mine = [p[0] for p in parts]
    assert sorted(mine[0] + mine[1]) == list(range(w.num_branches))
    assert len(mine[0]) == len(mine[1]) == 16  # 4 requests of 8 branches: two on each rank
    o = shard.gather_rows([torch.from_numpy(p[1]) for p in parts], mine, w).numpy()
    l = shard.gather_rows([torch.from_numpy(p[2]) for p in parts], mine, w).numpy()
    assert np.array_equal(o.reshape(-1, 128), ref_o) and np.array_equal(l.reshape(-1), ref_l)
    # no page is read by both ranks: the shares' unique KV adds up to the whole problem's
    assert parts[0][3] + parts[1][3] == oracle.unique_slots(w)[0]


def test_request_groups_follow_shared_pages():
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    assert shard.request_groups(W.make(5, small=True, values=False)) == [list(range(8 * i, 8 * i + 8)) for i in range(4)]
    # one shared prefix (and mounts across leaves) make one request
    for cfg in (2, 3, 4):
        assert len(shard.request_groups(W.make(cfg, small=True, values=False))) == 1
    with pytest.raises(ValueError):
        shard.request_assignment(W.make(2, small=True, values=False), 2)
    assert shard.head_range(8, 0, 3) == (0, 3) and shard.head_range(8, 2, 3) == (6, 8)
    with pytest.raises(ValueError):
        shard.head_range(2, 0, 4)


def _lse_merge(outs, lses):
    """Log-sum-exp merge of per-part (out, lse) in fp64 (test-side check of the split)."""
    lses = np.stack(lses)
    outs = np.stack(outs)
    M = lses.max(axis=0)
    fin = np.isfinite(M)
    w = np.where(np.isfinite(lses), np.exp(lses - np.where(fin, M, 0.0)), 0.0)
    L = w.sum(axis=0)
    out = np.where(fin[:, None], (w[..., None] * outs).sum(axis=0) / np.where(fin, L, 1.0)[:, None], 0.0)
    lse = np.where(fin, M + np.log(np.where(fin, L, 1.0)), -np.inf)
    return out, lse


def _seq_main(rank, world, port, out_dir):
    # one long shared prefix split by logical position: each rank the oracle's partial of its
    # range, then the all-gather the split needs (gloo) and the merge
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    dist.init_process_group("gloo")
    w = W.make(4, small=True)
    sub = shard.split_by_sequence(w, rank, world)
    o, l = oracle.fork_attn(sub, threads=max(1, oracle.threads_default() // world))
    ot, lt = torch.from_numpy(o), torch.from_numpy(l)
    go = [torch.empty_like(ot) for _ in range(world)]
    gl = [torch.empty_like(lt) for _ in range(world)]
    dist.all_gather(go, ot)
    dist.all_gather(gl, lt)
    if rank == 0:
        np.savez(os.path.join(out_dir, "seq.npz"), o=np.stack([x.numpy() for x in go]),
                 l=np.stack([x.numpy() for x in gl]))
    dist.barrier()
    dist.destroy_process_group()


def test_split_by_sequence_merges_to_the_whole_problem():
    import tempfile
    import oracle
    from shared_prefix_paged_attn_b300 import workloads as W
    with tempfile.TemporaryDirectory() as out:
        mp.start_processes(_seq_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        d = np.load(os.path.join(out, "seq.npz"))
    w = W.make(4, small=True)
    ref_o, ref_l = oracle.fork_attn(w)
    o, l = _lse_merge(list(d["o"]), list(d["l"]))
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_l))
    fin = ~np.isneginf(ref_l)
    assert np.abs(o[fin] - ref_o[fin]).max() < 1e-12 and np.abs(l[fin] - ref_l[fin]).max() < 1e-12


def test_sequence_split_is_a_partition_of_every_branch():
    from oracle import compact as C
    from shared_prefix_paged_attn_b300 import shard
    from shared_prefix_paged_attn_b300 import workloads as W
    w = W.make(3, small=True, values=False)
    for world in (1, 2, 3):
        parts = [shard.split_by_sequence(w, r, world) for r in range(world)]
        for b in range(w.num_branches):
            seen = np.concatenate([C.kept_indices(p, b) for p in parts])
            assert np.array_equal(np.sort(seen), C.kept_indices(w, b)) and len(set(seen.tolist())) == len(seen)
    cuts = shard.sequence_cuts(w, 4)
    assert cuts[0] == 0 and cuts[-1] == max(w.branch_len(b) for b in range(w.num_branches))
