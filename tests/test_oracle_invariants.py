"""Invariants of the optimum that follow from the definition of the placement problem.

Nest (Network- and Memory-Aware Device Placement) §4: the DP only adds options as
devices, memory, stages, candidate tiers or strategies are added, so the optimal
batch time can only fall; every stage of a plan holds at most its share of the
compute, so the bottleneck is bounded below by total compute over all devices;
a plan is rejected whenever its memory does not fit (§3.3).
"""
import numpy as np
import pytest

from memory_aware_device_gb300 import synth
from oracle import oracle as O


def _t(inst):
    r = O.solve(inst)
    return r["t_batch"] if r["status"] == 0 else None


def _le(a, b):
    """a <= b where None means infeasible (+infinity)."""
    return b is None or (a is not None and a <= b)


@pytest.mark.parametrize("seed", range(60))
def test_more_devices_never_hurt(seed):
    inst = synth.random_tiny(seed + 100, Lmax=6, Dmax=8)
    bigger = synth.random_tiny(seed + 100, Lmax=6, Dmax=8)
    bigger.D = inst.D * 2
    if int(bigger.tierG[-1]) < bigger.D:
        bigger.tierG = bigger.tierG.copy()
        bigger.tierG[-1] = int(bigger.tierG[-1]) * 2
        inst.tierG = bigger.tierG.copy()   # same tiers on both sides
    assert _le(_t(bigger), _t(inst))


@pytest.mark.parametrize("seed", range(60))
def test_more_memory_stages_candidates_strategies_never_hurt(seed):
    base = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
    t0 = _t(base)

    more_mem = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
    more_mem.budget = base.budget * 2 + 1000
    assert _le(_t(more_mem), t0)

    more_p = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
    more_p.Pmax = base.Pmax + 1
    more_p.M = max(base.M, more_p.Pmax)
    base_m = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
    base_m.M = more_p.M
    assert _le(_t(more_p), _t(base_m))

    if base.C < base.T:
        more_c = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
        extra = [t for t in range(base.T) if t not in set(base.cand.tolist())][0]
        more_c.cand = np.asarray(sorted(base.cand.tolist() + [extra]), np.int32)
        assert _le(_t(more_c), t0)

    more_s = synth.random_tiny(seed + 200, Lmax=6, Dmax=8)
    more_s.strat = np.concatenate([base.strat, np.asarray([[1, 1, 1, 0, 0], [2, 1, 1, 3, 1]],
                                                          np.int16)])
    assert _le(_t(more_s), t0)


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_bottleneck_lower_bound_total_compute(cfg):
    """v * D * R >= 3 sum(fl): each stage's replicas share its compute."""
    inst = synth.config_instance(cfg, 0)
    r = O.solve(inst)
    assert r["status"] == 0
    assert r["bottleneck"] * inst.D * inst.R >= 3 * int(inst.fl.sum())


def test_bound_is_tight_when_everything_else_is_free():
    # one strategy, all bytes and latency zero, R = 1, fl divisible: the bound is met
    L, D = 6, 8
    inst = synth.random_tiny(3)
    inst.L, inst.D, inst.unit = L, D, 1
    inst.fl = np.full(L, 8 * 1000, np.int64)
    for f in ("pd", "pe", "ao", "aw", "a2a"):
        setattr(inst, f, np.zeros(L, np.int64))
    inst.moe = np.zeros(L, np.uint8)
    inst.tierG = np.asarray([8], np.int64)
    inst.tierBw = np.asarray([1000], np.int64)
    inst.tierLat = np.asarray([0], np.int64)
    inst.cand = np.asarray([0], np.int32)
    inst.strat = np.asarray([[1, 1, 1, 0, 0]], np.int16)
    inst.R, inst.Pmax, inst.M, inst.budget = 1, 4, 100, 1 << 50
    r = O.solve(inst)
    assert r["bottleneck"] * D * inst.R == 3 * int(inst.fl.sum())


@pytest.mark.parametrize("seed", range(40))
def test_budget_monotone_and_zero_budget_infeasible(seed):
    inst = synth.random_tiny(seed + 400, Lmax=6, Dmax=8)
    ts = []
    for frac in (0.0, 0.25, 0.5, 1.0, 2.0, 8.0):
        inst.budget = int(5 * 10**6 * frac)
        ts.append(_t(inst))
    for a, b in zip(ts[1:], ts[:-1]):
        assert _le(a, b)
    # zero budget: infeasible unless the model holds no bytes at all
    if int(inst.pd.sum() + inst.pe.sum() + inst.aw.sum()) > 0 and inst.opt_factor >= 0:
        inst.budget = 0
        r = O.solve(inst)
        if int(inst.pd.sum() + inst.pe.sum()) > 0:
            assert r["status"] == 1


@pytest.mark.parametrize("cfg", [1, 2])
def test_every_returned_plan_fits_memory(cfg):
    """Recheck each stage of the plan against the §3.3 memory model at its position."""
    for b in range(min(4, synth.CONFIG_BATCH[cfg])):
        inst = synth.config_instance(cfg, b)
        r = O.solve(inst)
        P = len(r["plan"])
        for q, (i, j, k, s, c) in enumerate(r["plan"]):
            t = O.terms(inst, i, j, k.bit_length() - 1, s)
            pos = P - q
            assert t["stat"] + (pos - 1) * t["stash"] <= inst.budget


def test_deterministic():
    inst = synth.config_instance(2, 3)
    a = O.solve(inst, want_dp=True)
    b = O.solve(inst, want_dp=True)
    assert a["plan"] == b["plan"] and (a["dp"] == b["dp"]).all()
