"""Pins for the joint microbatch-size search.

Nest (Network- and Memory-Aware Device Placement) §5.2.3 explores the microbatch
size together with the placement.  A variant with b samples per microbatch scales
every per-microbatch quantity by b and runs M = 4096 / b microbatches, so the
iteration covers the same 4096 samples; t_batch = bottleneck x (M + p - 1) then
compares variants directly.  Pinned by two closed forms that pull in opposite
directions - with pure compute a plan's bottleneck scales with b and the bubble
(p - 1) b grows, so b = 1 is optimal; with pure per-microbatch latency the
bottleneck does not scale and fewer, larger microbatches win, so b = 8 is optimal -
and by the memory model (activations grow with b, so a stage's pmax never grows).
"""
import copy

import numpy as np
import pytest

from memory_aware_device_gb300 import synth
from oracle import oracle as O


def test_variants_scale_per_microbatch_quantities_only():
    x = synth.config_instance(4, 3)
    for b in synth.MICROBATCH_SIZES:
        y = synth.microbatch_variant(x, b)
        for f in ("fl", "ao", "aw", "a2a"):
            assert (getattr(y, f) == b * getattr(x, f)).all()
        for f in ("pd", "pe", "moe", "tierG", "tierBw", "tierLat", "cand", "strat"):
            assert (getattr(y, f) == getattr(x, f)).all()
        assert y.M * b == synth.GLOBAL_BATCH and y.budget == x.budget


def test_single_size_is_the_plain_solve():
    x = synth.config_instance(1, 0)
    j = O.solve_joint([synth.microbatch_variant(x, 1)])
    assert j["best"] == 0 and j["t_batch"] == O.solve(x)["t_batch"]


def _compute_only(seed):
    rng = np.random.default_rng(seed)
    x = synth.random_tiny(seed, Lmax=6, Dmax=8)
    L = x.L
    x.fl = rng.integers(1, 50, size=L).astype(np.int64) * 4096   # exact divisions
    x.R = 1
    for f in ("pd", "pe", "ao", "aw", "a2a"):
        setattr(x, f, np.zeros(L, np.int64))
    x.moe = np.zeros(L, np.uint8)
    x.tierLat = np.zeros_like(x.tierLat)
    x.tierBw = np.full_like(x.tierBw, 1 << 40)
    x.budget = 1 << 60
    x.strat = np.array([[1, 1, 1, 0, 0]], np.int16)
    x.M = synth.GLOBAL_BATCH
    return x


@pytest.mark.parametrize("seed", range(30))
def test_pure_compute_prefers_the_smallest_microbatch(seed):
    x = _compute_only(seed)
    j = O.solve_joint(synth.joint_batch([x]))
    ts = [r["t_batch"] for r in j["results"]]
    assert j["best"] == 0 and ts[0] == min(ts)
    # a plan's bottleneck scales with b, so no variant beats b = 1 on the same plan
    assert all(t >= ts[0] for t in ts)


def test_pure_latency_prefers_the_largest_microbatch():
    # no compute, one byte of activation per sample, tensor parallelism of 2: every
    # microbatch pays the same all-reduce latencies whatever its size, so fewer, larger
    # microbatches win (the bandwidth term adds at most a nanosecond per collective)
    checked = 0
    for seed in range(60):
        x = _compute_only(seed)
        if x.D < 2:
            continue
        x.fl = np.zeros(x.L, np.int64)
        x.ao = np.ones(x.L, np.int64)
        x.tierLat = np.full_like(x.tierLat, 100000)
        x.strat = np.array([[2, 1, 1, 0, 0]], np.int16)
        j = O.solve_joint(synth.joint_batch([x]))
        ts = [r["t_batch"] for r in j["results"]]
        assert all(r["status"] == 0 for r in j["results"])
        assert j["best"] == len(ts) - 1 and ts == sorted(ts, reverse=True), ts
        checked += 1
    assert checked >= 20


@pytest.mark.parametrize("seed", range(20))
def test_larger_microbatches_never_fit_more_positions(seed):
    x = synth.random_tiny(seed + 900, Lmax=5, Dmax=8)
    K = (x.D // x.unit).bit_length()
    vs = [synth.microbatch_variant(x, b) for b in synth.MICROBATCH_SIZES]
    for i in range(x.L):
        for jj in range(i + 1, x.L + 1):
            for m in range(K):
                for s in range(len(x.strat)):
                    pm = [O.terms(v, i, jj, m, s)["pmax"] for v in vs]
                    assert all(a >= b for a, b in zip(pm, pm[1:])), (i, jj, m, s, pm)


def test_joint_is_the_best_variant():
    for cfg, b in ((2, 0), (2, 5), (4, 1)):
        x = synth.config_instance(cfg, b)
        j = O.solve_joint(synth.joint_batch([x]))
        solved = [r["t_batch"] for r in j["results"] if r["status"] == 0]
        assert j["t_batch"] == min(solved)
        assert j["results"][j["best"]]["t_batch"] == j["t_batch"]
