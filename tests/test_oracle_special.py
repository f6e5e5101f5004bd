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


def test_batch_time_ties_go_to_fewer_stages():
    """Two plans with the same batch time: one stage on both devices (6 compute + 3
    amortised gradient AllReduce, times M = 2) and a two-stage pipeline of one device
    each (6, times M + 1 = 3): 18 ns both.  The tie goes to fewer stages."""
    import brute
    inst = make(L=2, fl=(2, 2), pd=(3, 3), D=2, G=(2,), bw=(1000,), lat=(0,), Pmax=2, M=2)
    plans = sorted((t, P, v) for t, P, v, _ in brute.enumerate_plans(inst, O.cost_tensor(inst), O.links(inst)))
    assert plans[:2] == [(18, 1, 9), (18, 2, 6)]
    r = O.solve(inst)
    assert (r["t_batch"], r["bottleneck"], len(r["plan"])) == (18, 9, 1)
    assert r["plan"][0][:3] == (0, 2, 2)


@pytest.mark.parametrize("heavy", [0, 1])
def test_stage_times_at_the_cap_are_infeasible(heavy):
    """Stage times (load plus link costs) of 2^40 - 1 ns or more are infeasible.  Two
    layers whose activations fit one at a time but not together, so the only plans
    are two one-device stages; the heavy layer's compute plus the 3 ns link lands on
    the cap exactly, or one below it."""
    CAP = (1 << 40) - 1
    for link, ok in ((3, False), (2, True)):
        fl = [0, 0]
        fl[heavy] = (CAP - 3) // 3        # compute 3 fl = 2^40 - 4
        inst = make(L=2, fl=fl, ao=(link, 0), aw=(1, 2), D=2, G=(2,), bw=(1000,), lat=(0,),
                    Pmax=2, M=2, budget=2, opt=0)
        assert O.terms(inst, 0, 2, 0, 0)["pmax"] == 0          # both layers: 3 bytes > 2
        r = O.solve(inst)
        if ok:
            assert r["status"] == 0 and r["bottleneck"] == CAP - 3 + link
            assert r["t_batch"] == (CAP - 3 + link) * 3 and len(r["plan"]) == 2
        else:
            assert r["status"] == 1
            if heavy:   # the last stage's own cell holds no value at the cap either
                dp = O.solve(inst, want_dp=True)["dp"]
                assert (dp[1] == O.INF).all()


def test_a_stage_load_at_the_cap_is_infeasible():
    """A one-stage plan whose compute alone is 2^40 - 1 ns has no feasible load; one
    flop less per pass gives 2^40 - 4 ns, which is feasible."""
    CAP = (1 << 40) - 1
    for fl, ok in ((CAP // 3, False), (CAP // 3 - 1, True)):
        inst = make(fl=fl, D=1, G=(1,))
        assert (O.cost_tensor(inst)[0, 0, 0] == O.INF) != ok
        r = O.solve(inst)
        assert (r["status"], r["t_batch"]) == ((0, CAP - 3) if ok else (1, -1))
