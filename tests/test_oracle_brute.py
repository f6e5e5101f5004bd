"""Pin the oracle's dynamic program to exhaustive enumeration of every plan.

Nest (Network- and Memory-Aware Device Placement) claims its DP is optimal
without enumerating placements (§4, Eq. 3 and the worked example of Fig. 4);
the optimum is therefore the minimum over ALL plans, which `brute.py` enumerates.
"""
import pytest

import brute
from memory_aware_device_gb300 import synth
from oracle import oracle as O


def _check(inst):
    w = O.cost_tensor(inst)
    X = O.links(inst)
    b = brute.brute_optimum(inst, w, X)
    r = O.solve(inst)
    if b is None:
        assert r["status"] == 1 and r["t_batch"] == -1 and r["plan"] == []
        return None
    assert r["status"] == 0
    assert (r["t_batch"], len(r["plan"]), r["bottleneck"]) == b
    # the returned plan is itself feasible and achieves the optimum
    assert brute.price_plan(inst, w, X, r["plan"]) == (b[0], b[2])
    return b


@pytest.mark.parametrize("chunk", range(8))
def test_random_tiny_instances(chunk):
    stages = set()
    for seed in range(chunk * 250, (chunk + 1) * 250):
        inst = synth.random_tiny(seed, Lmax=7, Dmax=16)
        b = _check(inst)
        if b is not None:
            stages.add(b[1])
    # the sample must exercise multi-stage plans, not just single stages
    assert max(stages) >= 3


def test_workload_1_exhaustive():
    inst = synth.config_instance(1, 0)
    assert _check(inst) is not None


def test_multi_stage_workload_1_variants():
    """Workload 1 with tighter memory forces pipelines; still equal to brute force."""
    base = synth.config_instance(1, 0)
    seen = set()
    for budget in (3 * 10**8, 6 * 10**8, 10**9, 2 * 10**9, 4 * 10**9):
        base.budget = budget
        b = _check(base)
        if b:
            seen.add(b[1])
    assert len(seen) >= 2
