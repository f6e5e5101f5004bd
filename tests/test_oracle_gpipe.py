"""Pins for the GPipe stash rule of the oracle.

Nest (Network- and Memory-Aware Device Placement) §3.3: the stashed microbatches of
a stage are (s - 1) at position s from the pipeline end under 1F1B and scale with
B/d under GPipe.  Read here as: each of the q data-parallel replicas runs
ceil(M / q) of the M microbatches and holds all of them at once, at every
position.  Pinned by (1) the defining property, feasibility independent of the
position; (2) the 1F1B rule, itself pinned by a linear scan of Mem(S, p): a GPipe
stage fits exactly when the same stage fits at 1F1B position ceil(M / q) + 1,
which holds the same number of stashed microbatches; (3) exhaustive enumeration of
plans; (4) more stash never helps.
"""
import copy

import numpy as np
import pytest

import brute
from memory_aware_device_gb300 import synth
from oracle import oracle as O


def gpipe(x):
    y = copy.deepcopy(x)
    y.schedule = 1
    return y


def _tuples(x):
    K = (x.D // x.unit).bit_length()
    for i in range(x.L):
        for j in range(i + 1, x.L + 1):
            for m in range(K):
                for s in range(len(x.strat)):
                    yield i, j, m, s


@pytest.mark.parametrize("seed", range(40))
def test_feasibility_is_position_independent(seed):
    x = gpipe(synth.random_tiny(seed, Lmax=5, Dmax=16))
    assert O.validate(x) == 0
    for i, j, m, s in _tuples(x):
        t = O.terms(x, i, j, m, s)
        if t["valid"]:
            assert t["pmax"] in (0, x.Pmax)


def test_gpipe_equals_1f1b_at_the_same_stash_count():
    # M = 32 microbatches, Pmax = 31: for q >= 2 a GPipe replica holds
    # ceil(32 / q) <= 16 microbatches, which 1F1B position ceil(32 / q) + 1 <= 17 holds too
    checked = 0
    for seed in range(60):
        x = synth.random_tiny(seed, Lmax=5, Dmax=16)
        x.M, x.Pmax = 32, 31
        g = gpipe(x)
        for i, j, m, s in _tuples(x):
            t1, tg = O.terms(x, i, j, m, s), O.terms(g, i, j, m, s)
            assert t1["valid"] == tg["valid"]
            if not t1["valid"]:
                continue
            t, cp = int(x.strat[s][0]), int(x.strat[s][1])
            q = (x.unit << m) // (t * cp)
            if q < 2:
                continue
            n = -(-x.M // q)
            assert (tg["pmax"] == x.Pmax) == (t1["pmax"] >= n + 1), (seed, i, j, m, s, q, t1, tg)
            assert tg["tau"] == t1["tau"]          # the schedule changes memory only
            checked += 1
    assert checked > 1000


@pytest.mark.parametrize("chunk", range(4))
def test_gpipe_dp_matches_exhaustive_enumeration(chunk):
    for seed in range(chunk * 150, (chunk + 1) * 150):
        x = gpipe(synth.random_tiny(seed + 50000, Lmax=7, Dmax=16))
        w, X = O.cost_tensor(x), O.links(x)
        b = brute.brute_optimum(x, w, X)
        r = O.solve(x)
        if b is None:
            assert r["status"] == 1
            continue
        assert r["status"] == 0 and (r["t_batch"], len(r["plan"]), r["bottleneck"]) == b
        assert brute.price_plan(x, w, X, r["plan"]) == (b[0], b[2])


@pytest.mark.parametrize("seed", range(60))
def test_more_stash_never_helps(seed):
    # with M / q >= Pmax - 1 for every strategy, GPipe stashes at least as much as any
    # 1F1B position, so its optimum can only be worse (or infeasible)
    x = synth.random_tiny(seed + 7000, Lmax=7, Dmax=16)
    qmax = x.D // min(int(t) * int(cp) for t, cp, *_ in x.strat)
    x.M = max(x.M, qmax * max(x.Pmax - 1, 1))
    r1, rg = O.solve(x), O.solve(gpipe(x))
    if r1["status"] == 1:
        assert rg["status"] == 1
    elif rg["status"] == 0:
        assert rg["t_batch"] >= r1["t_batch"]


def test_workload_variant_solves():
    # with all 4096 microbatches of an iteration in flight GPipe does not fit; with 512
    # it does, and every stage of the plan fits at every position
    x = gpipe(synth.config_instance(2, 0))
    assert O.solve(x)["status"] == 1
    x.M = 512
    r = O.solve(x)
    assert r["status"] == 0
    w = O.cost_tensor(x)
    for i, j, k, s, _ in r["plan"]:
        m = (k // x.unit).bit_length() - 1
        assert int(w[i * x.L - i * (i - 1) // 2 + (j - i - 1)][m][s]) & 0xFF == x.Pmax


def test_invalid_schedule_rejected():
    x = synth.random_tiny(1)
    x.schedule = 2
    assert O.validate(x) == 2
