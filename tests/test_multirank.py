"""Multi-rank host logic on CPU (gloo, world size 2): the trees of N
GRPO-shaped batches are split over the ranks by KK balancing of their
ancestor pairs (every sequence on exactly one rank, loads close), and the
job totals are the summed work over the slowest rank's time.  The GPU data
path of each rank is the single-GPU path and needs no collective."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import prefix_shared_tree_attention_gb300 as tpa
        seqs = bench.rank_sequences(rank, world, tpa)
        gathered = [None] * world
        dist.all_gather_object(gathered, [tuple(s) for s in seqs])
        red = bench.reduce_job(1.0e12 * (rank + 1), 100 * (rank + 1), 10.0 + rank)
        if rank == 0:
            q.put((gathered, red))
    finally:
        dist.destroy_process_group()


def test_two_ranks_split_trees_and_reduce():
    import torch.multiprocessing as mp

    import prefix_shared_tree_attention_gb300 as tpa
    from synth import CONFIGS, make_sequences
    tpa.lib()  # build once in this process before the workers load it
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        gathered, (flops, rows, ms) = q.get(timeout=600)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert flops == pytest.approx(3.0e12) and rows == 300 and ms == pytest.approx(11.0)
    everything = sorted(tuple(s) for r in range(2) for s in make_sequences(2, seed=2 + 1000 * r))
    assert sorted(gathered[0] + gathered[1]) == everything  # a partition of both batches
    mb = CONFIGS[2].max_tokens_per_mb
    loads = [int(tpa.tree_pack([list(s) for s in g], mb).info.ancestor_pairs) for g in gathered]
    assert min(loads) > 0 and (max(loads) - min(loads)) / max(loads) < 0.25
