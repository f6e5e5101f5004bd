"""Special cases of the placement DP that reduce to textbook problems.

With free communication, unlimited memory and one strategy, a pipeline of
width-1 stages is the chains-on-chains partition problem (split a sequence into
p contiguous blocks minimising the largest block sum), solved here by binary
search on the bound plus greedy packing, an algorithm independent of the DP.
The DP's objective is Nest (Network- and Memory-Aware Device Placement)
Appendix K Algorithm 1: bottleneck stage time x (M + p - 1).
"""
import json
import os

import numpy as np
import pytest

from helpers import make
from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def greedy_blocks(w, bound):
    """Blocks needed when packing w left to right under the bound (None if an element exceeds it)."""
    blocks, cur = 1, 0
    for x in w:
        if x > bound:
            return None
        if cur + x > bound:
            blocks, cur = blocks + 1, x
        else:
            cur += x
    return blocks


def chains_optimum(w, p):
    """Smallest bound with a partition into at most p blocks (binary search + greedy)."""
    lo, hi = max(w), sum(w)
    while lo < hi:
        mid = (lo + hi) // 2
        n = greedy_blocks(w, mid)
        if n is not None and n <= p:
            hi = mid
        else:
            lo = mid + 1
    return lo


def test_chains_golden():
    g = json.load(open(os.path.join(GOLD, "chains_on_chains.json")))
    for p, want in g["optimum"].items():
        assert chains_optimum(g["w"], int(p)) == want


def chains_instance(w, D, Pmax, M):
    """Width-1 pipelines only: the link tier holds 2 devices, so every stage next
    to a link has k = 1; a lone stage may use any width.  Zero bytes and zero
    latency make every collective and link free; R = 1 makes a layer cost 3 fl."""
    top = 1
    while top < D:
        top *= 2
    G = (2, max(top, 4))
    return make(L=len(w), fl=np.asarray(w, np.int64), G=G, bw=(1000, 1000), lat=(0, 0),
                cand=(0,), D=D, Pmax=Pmax, M=M, R=1, opt=0)


def expected_chains(w, D, Pmax, M):
    best = None
    k = 1
    while k <= D:  # one stage of width k: ceil(3 sum / k) per microbatch
        t = M * -(-3 * sum(w) // k)
        best = t if best is None else min(best, t)
        k *= 2
    for p in range(2, min(Pmax, D, len(w)) + 1):
        best = min(best, (M + p - 1) * 3 * chains_optimum(w, p))
    return best


def test_chains_golden_through_dp():
    g = json.load(open(os.path.join(GOLD, "chains_on_chains.json")))
    w = g["w"]
    # D = 8 devices, up to 8 stages, M = 8: a p-stage pipeline costs (7 + p) * 3 * B(p)
    # with B(p) from the hand-worked table; one stage of width k costs 8 * ceil(93 / k)
    inst = chains_instance(w, D=8, Pmax=8, M=8)
    r = O.solve(inst)
    assert r["status"] == 0
    assert r["t_batch"] == expected_chains(w, 8, 8, 8)


@pytest.mark.parametrize("seed", range(40))
def test_chains_random(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(2, 13))
    w = [int(x) for x in rng.integers(0, 1000, size=L)]
    D = int(rng.integers(3, 13))
    Pmax = int(rng.integers(2, 9))
    M = int(rng.integers(Pmax, 3 * Pmax + 60))
    inst = chains_instance(w, D, Pmax, M)
    r = O.solve(inst)
    assert r["status"] == 0
    assert r["t_batch"] == expected_chains(w, D, Pmax, M)
    if len(r["plan"]) > 1:
        # every stage of a pipeline is one device wide and within the chains bound
        bound = chains_optimum(w, len(r["plan"]))
        for (i, j, k, s, c) in r["plan"]:
            assert k == 1
            assert 3 * sum(w[i:j]) <= 3 * bound


@pytest.mark.parametrize("seed", range(20))
def test_single_stage_closed_form(seed):
    """Pmax = 1: t_batch = M * min over widths and strategies of the stage time."""
    from memory_aware_device_gb300 import synth
    inst = synth.random_tiny(seed + 7000, Lmax=6, Dmax=16)
    inst.Pmax = 1
    r = O.solve(inst)
    best = None
    m = 0
    while (1 << m) <= inst.D // inst.unit:
        for s in range(inst.S):
            t = O.terms(inst, 0, inst.L, m, s)
            if t["valid"] and t["tau"] < O.CAP and t["pmax"] >= 1:
                best = t["tau"] if best is None else min(best, t["tau"])
        m += 1
    if best is None:
        assert r["status"] == 1
    else:
        assert r["status"] == 0 and r["t_batch"] == inst.M * best and len(r["plan"]) == 1


def test_one_unit_means_one_stage():
    from memory_aware_device_gb300 import synth
    for seed in range(30):
        inst = synth.random_tiny(seed + 9000)
        inst.D = inst.unit
        inst.tierG = np.asarray(sorted(set([max(int(g), 1) for g in inst.tierG])), np.int64)
        r = O.solve(inst)
        if r["status"] == 0:
            assert len(r["plan"]) == 1 and r["plan"][0][2] == inst.unit
