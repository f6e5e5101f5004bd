"""The multi-GPU path is replicas over independent instances: each rank solves its own
batch and only the timing is combined.  These tests run that host logic as two gloo
ranks on the CPU: disjoint shards, whole-job units summed, job time the slowest rank's,
and the rank results equal to solving every instance alone (nothing is exchanged)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from memory_aware_device_gb300 import synth  # noqa: E402


def _fingerprint(x):
    """Everything that defines an instance, as bytes."""
    return b"|".join([repr((x.L, x.D, x.unit, x.Pmax, x.R, x.M, x.budget, x.opt_factor)).encode()] +
                     [a.tobytes() for a in (x.fl, x.pd, x.pe, x.ao, x.aw, x.a2a, x.moe, x.tierG, x.tierBw,
                                            x.tierLat, x.cand, x.strat)])


def _rank(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        insts = bench.rank_instances(2, rank)
        units = sum(bench.relaxations(x) for x in insts)
        local_ms = 10.0 + 5.0 * rank               # the second rank is slower
        job_units, job_ms = bench.job_totals(units, local_ms, dist)
        from oracle import oracle as O
        res = [O.solve(x)["t_batch"] for x in insts[:2]]
        q.put((rank, [_fingerprint(x) for x in insts], units, job_units, job_ms, res))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_aggregate():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    out = sorted(q.get() for _ in range(2))
    (r0, fl0, u0, ju0, jm0, res0), (r1, fl1, u1, ju1, jm1, res1) = out
    assert (r0, r1) == (0, 1)
    assert len(fl0) == len(fl1) == synth.CONFIG_BATCH[2]
    assert not set(fl0) & set(fl1), "ranks must solve different instances"
    assert ju0 == ju1 == u0 + u1                   # whole-job units
    assert jm0 == jm1 == 15.0                      # the slowest rank's time
    # nothing is exchanged: a rank's results are those of its instances solved alone
    from oracle import oracle as O
    alone = [O.solve(x)["t_batch"] for x in bench.rank_instances(2, 1)[:2]]
    assert res1 == alone


def test_single_process_totals_are_local():
    assert bench.job_totals(7.0, 3.0) == (7.0, 3.0)


def test_tiny_workload_is_the_same_instance_on_every_rank():
    a, b = bench.rank_instances(1, 0), bench.rank_instances(1, 3)
    assert len(a) == len(b) == 1 and _fingerprint(a[0]) == _fingerprint(b[0])
