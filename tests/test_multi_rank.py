"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The verify step partitions by sequence with no data exchange: each rank draws
its own batch and the job rate is all ranks' tokens over the slowest rank's
time.  These checks run the same helpers bench.py uses, in two gloo ranks.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    import oracle
    seed = bench.rank_seed(7, rank)
    w = workloads.generate("tiny_tree_fp32", seed=seed)
    # the rank's own work: the oracle's step on its own batch
    att = oracle.tree_attn(w)
    am, alen, path, nxt = oracle.accept_greedy(w["tree_tokens"], w["logits"], "f32", w["tree_parents"], 3)
    local_ms = 1.0 + rank            # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, world)
    rate = bench.whole_job_rate(w["B"] * w["T"], world, ms)
    gathered = [None] * world
    dist.all_gather_object(gathered, (seed, float(att.sum()), ms, rate, int(alen[0])))
    if rank == 0:
        out.put(gathered)
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_sequence_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (s0, a0, ms0, r0, _), (s1, a1, ms1, r1, _) = res
    assert s0 != s1 and a0 != a1          # independent batches
    assert ms0 == ms1 == 2.0              # both ranks report the slowest time
    assert r0 == r1 == pytest.approx(2 * 7 / 2.0e-3)
