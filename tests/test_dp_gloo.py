"""Row-sharded (data-parallel) host logic, on CPU with two gloo ranks.

Each rank samples its own shard of one batch with the CPU oracle (and
verifies its share of a batch of draft trees); the gathered tokens must equal
those of the whole batch at once (rows and requests are independent and their
noise is keyed by their ids, so the data path needs no collective), and the
elapsed time reduction is the maximum over ranks, as the benchmark reports it.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle as O
from speculative_verification_gb300 import dp as DP
from speculative_verification_gb300 import workloads as W
from tests.parity import subset_sample, subset_tree

ROWS = 10


def _batch():
    return W.make(2, rows=ROWS)


def _trees():
    return W.tree(seed=8, requests=7, vocab=3000, max_nodes=6)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _batch()
        start, stop = DP.shard_rows(w["num_rows"], rank, world)
        shard = subset_sample(w, list(range(start, stop)))
        shard["row_id"] = np.arange(start, stop, dtype=np.uint32)  # the rows' ids in the whole batch
        ref = O.process_sample(shard)
        tokens = [None] * world
        dist.all_gather_object(tokens, (start, stop, ref["token"].tolist(), ref["status"].tolist()))
        # draft trees, split by request the same way
        tw = _trees()
        t0, t1 = DP.shard_rows(tw["num_requests"], rank, world)
        tshard = subset_tree(tw, list(range(t0, t1)))
        tshard["row_id"] = np.arange(t0, t1, dtype=np.uint32)
        tref = O.tree_verify(tshard)
        trees = [None] * world
        dist.all_gather_object(trees, (t0, t1, tref["out_tokens"].tolist(), tref["out_path"].tolist()))
        t = torch.tensor([10.0 * (rank + 1)])  # a stand-in elapsed time per rank
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        seeds = [None] * world
        dist.all_gather_object(seeds, [DP.ring_seed(2, rank, i) for i in range(4)])
        if rank == 0:
            np.save(os.path.join(out_dir, "gathered.npy"), np.array(tokens, dtype=object), allow_pickle=True)
            np.save(os.path.join(out_dir, "trees.npy"), np.array(trees, dtype=object), allow_pickle=True)
            np.save(os.path.join(out_dir, "tmax.npy"), t.numpy())
            np.save(os.path.join(out_dir, "seeds.npy"), np.array(seeds))
    finally:
        dist.destroy_process_group()


def test_shard_rows_partition():
    for n in (0, 1, 7, 64, 65):
        for world in (1, 2, 3, 8):
            spans = [DP.shard_rows(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        DP.shard_rows(8, 2, 2)


def test_aggregate_rate():
    assert DP.aggregate_rate(64, 100, 4, 1000.0) == pytest.approx(64 * 100 * 4)
    with pytest.raises(ValueError):
        DP.aggregate_rate(64, 1, 1, 0.0)


def test_two_gloo_ranks_match_whole_batch(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    gathered = np.load(tmp_path / "gathered.npy", allow_pickle=True)
    whole = O.process_sample(_batch())
    tok = np.full(ROWS, -2, np.int64)
    st = np.full(ROWS, -2, np.int64)
    for start, stop, t, s in gathered:
        tok[start:stop] = t
        st[start:stop] = s
    assert np.array_equal(tok, whole["token"]) and np.array_equal(st, whole["status"])
    trees = np.load(tmp_path / "trees.npy", allow_pickle=True)
    whole_t = O.tree_verify(_trees())
    R = int(whole_t["num_accepted"].size)
    got_tok = np.full(whole_t["out_tokens"].shape, -2, np.int64)
    got_path = np.full(whole_t["out_path"].shape, -2, np.int64)
    for t0, t1, tt, pp in trees:
        got_tok[t0:t1] = tt
        got_path[t0:t1] = pp
    assert np.array_equal(got_tok, whole_t["out_tokens"]) and np.array_equal(got_path, whole_t["out_path"])
    assert R == 7 and (whole_t["num_accepted"] > 0).any()
    assert float(np.load(tmp_path / "tmax.npy")[0]) == 20.0
    seeds = np.load(tmp_path / "seeds.npy")
    assert len(np.unique(seeds)) == seeds.size  # every rank samples its own batches


_RANK_SCRIPT = r"""
import os, sys
import torch
import torch.distributed as dist
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
assert rank == int(os.environ["RANK"]) == int(os.environ["LOCAL_RANK"])
if len(sys.argv) > 2 and int(sys.argv[2]) == rank:
    sys.exit(3)  # this rank fails before the collective
t = torch.tensor([float(rank + 1)])
dist.all_reduce(t)
with open(os.path.join(sys.argv[1], "rank%d" % rank), "w") as f:
    f.write("%d %d %.0f" % (rank, world, t.item()))
dist.destroy_process_group()
"""


def test_launch_local_starts_every_rank(tmp_path):
    """bench.py --gpus N without torchrun starts its ranks with
    DP.launch_local: every rank gets torchrun's variables, joins the same
    process group and exits 0."""
    import sys
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT)
    world = 3
    assert DP.launch_local(world, [sys.executable, str(script), str(tmp_path)], timeout=300) == 0
    for r in range(world):
        rank, w, total = (tmp_path / ("rank%d" % r)).read_text().split()
        assert (int(rank), int(w), int(total)) == (r, world, world * (world + 1) // 2)


def test_launch_local_reports_a_failed_rank(tmp_path):
    """A rank that exits non-zero: the launcher returns its code and stops the
    rank left waiting in the collective."""
    import sys
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT)
    assert DP.launch_local(2, [sys.executable, str(script), str(tmp_path), "1"], timeout=300) == 3
    assert not (tmp_path / "rank1").exists()
