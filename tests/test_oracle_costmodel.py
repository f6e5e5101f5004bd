"""Pin the oracle's stage-cost model (load() of Nest §4 and the §3.3 memory model).

Each test isolates one term by zeroing every other input and compares it with a
closed form from the literature the pages build on:
  - ring collectives (Thakur, Rabenseifner & Gropp 2005; Patarasuk & Yuan 2009):
    AllReduce over n devices takes 2(n-1) latency steps and moves 2(n-1)/n of the
    buffer per device; AllGather, ReduceScatter and AllToAll take (n-1) steps and
    move (n-1)/n of it;
  - Megatron-LM tensor parallelism (Shoeybi et al. 2019): two AllReduces forward
    and two backward per transformer layer;
  - GShard expert parallelism (Lepikhin et al. 2020): dispatch and combine
    AllToAll in the forward pass and again in the backward pass;
  - ZeRO (Rajbhandari et al. 2020): per-device model-state bytes of the Figure 1
    worked example, and 1.5x the data-parallel traffic at stage 3;
  - backward pass = 2x forward flops, recompute adds one forward pass.
Values are chosen so that every ceiling is exact, so the closed forms hold with
plain rational arithmetic.
"""
import json
import os
from fractions import Fraction as F

import numpy as np
import pytest

from helpers import BIG, make
from memory_aware_device_gb300 import synth
from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def ring_allreduce(n, V, alpha, beta):
    return 2 * (n - 1) * alpha + F(2 * (n - 1), n) * V * 1000 / beta


def ring_gather(n, V, alpha, beta):  # AllGather / ReduceScatter / AllToAll
    return (n - 1) * alpha + F(n - 1, n) * V * 1000 / beta


def test_compute_three_passes():
    inst = make(fl=10**9, R=10**6, strat=((1, 1, 1, 0, 0), (1, 1, 1, 0, 1)))
    assert O.terms(inst, 0, 1, 0, 0)["tau"] == 3000   # forward + 2x backward
    assert O.terms(inst, 0, 1, 0, 1)["tau"] == 4000   # + recomputed forward


def test_compute_splits_over_replicas_and_tp():
    # 8 devices: TP 2 x DP 4; no bytes at all, so only compute remains
    inst = make(fl=8 * 10**9, R=10**6, strat=((2, 1, 1, 0, 0),))
    assert O.terms(inst, 0, 1, 3, 0)["tau"] == 3 * 8 * 10**9 // 10**6 // 8


def test_tensor_parallel_four_allreduces():
    n, A, alpha, beta = 4, 8 * 10**6, 1000, 10**6
    inst = make(ao=A, G=(8,), bw=(beta,), lat=(alpha,), strat=((4, 1, 1, 0, 0),))
    t = O.terms(inst, 0, 1, 2, 0)   # k = 4 = t, so q = 1
    assert t["tp"] == 4 * ring_allreduce(n, A, alpha, beta)
    assert t["tau"] == t["tp"]


def test_tensor_parallel_uses_smallest_covering_tier():
    # TP over 4 devices does not fit a 2-device tier: the 8-device tier's link is used
    n, A = 4, 8 * 10**6
    inst = make(ao=A, G=(2, 8), bw=(10**7, 2 * 10**6), lat=(10, 700), strat=((4, 1, 1, 0, 0),))
    assert O.terms(inst, 0, 1, 2, 0)["tp"] == 4 * ring_allreduce(n, A, 700, 2 * 10**6)
    inst2 = make(ao=A, G=(4, 8), bw=(10**7, 2 * 10**6), lat=(10, 700), strat=((4, 1, 1, 0, 0),))
    assert O.terms(inst2, 0, 1, 2, 0)["tp"] == 4 * ring_allreduce(n, A, 10, 10**7)


def test_gradient_allreduce_amortised_over_iteration():
    n, P, alpha, beta, M = 8, 8 * 10**6, 500, 10**6, 7
    inst = make(pd=P, G=(8,), bw=(beta,), lat=(alpha,), M=M, strat=((1, 1, 1, 0, 0),))
    t = O.terms(inst, 0, 1, 3, 0)
    assert t["sd"] == ring_allreduce(n, P, alpha, beta)
    assert t["tau"] == t["sd"] / M


def test_zero3_traffic_is_one_and_a_half_times_data_parallel():
    # each of n replicas runs one microbatch (M = n); no latency
    n, P, beta = 8, 8 * 10**6, 10**6
    strat = ((1, 1, 1, 0, 0), (1, 1, 1, 3, 0))
    inst = make(pd=P, G=(8,), bw=(beta,), lat=(0,), M=n, strat=strat)
    base, z3 = O.terms(inst, 0, 1, 3, 0), O.terms(inst, 0, 1, 3, 1)
    iter_base = n * base["tau"]
    iter_z3 = n * z3["tau"]
    assert F(iter_z3, iter_base) == F(3, 2)
    # gathers before forward and before backward, and a ReduceScatter of gradients
    assert z3["z3"] == ring_gather(n, 2 * P, 0, beta)
    assert z3["sd"] == ring_gather(n, P, 0, beta)


def test_zero12_sync_matches_allreduce_volume():
    n, P, alpha, beta = 8, 8 * 10**6, 300, 10**6
    strat = ((1, 1, 1, 0, 0), (1, 1, 1, 1, 0), (1, 1, 1, 2, 0))
    inst = make(pd=P, G=(8,), bw=(beta,), lat=(alpha,), M=1, strat=strat)
    sd = [O.terms(inst, 0, 1, 3, s)["sd"] for s in range(3)]
    # ReduceScatter + AllGather has the same latency steps and bytes as AllReduce
    assert sd[0] == sd[1] == sd[2] == ring_allreduce(n, P, alpha, beta)


def test_zero_memory_figure1_worked_example():
    g = json.load(open(os.path.join(GOLD, "zero_memory.json")))
    psi, nd = g["psi"], g["n_d"]
    strat = tuple((1, 1, 1, z, 0) for z in range(4))
    inst = make(pd=2 * psi, D=64, G=(64,), bw=(10**6,), lat=(0,), opt=g["K"] // 2, strat=strat)
    m = nd.bit_length() - 1
    stat = [O.terms(inst, 0, 1, m, z)["stat"] for z in range(4)]
    want = g["bytes_per_device"]
    assert stat == [want["baseline"], want["P_os"], want["P_os+g"], want["P_os+g+p"]]


def test_expert_alltoall_four_per_moe_layer():
    n, V, alpha, beta = 8, 16 * 10**6, 200, 4 * 10**6
    inst = make(a2a=V, moe=1, G=(8,), bw=(beta,), lat=(alpha,), strat=((1, 1, 8, 0, 0),))
    t = O.terms(inst, 0, 1, 3, 0)    # k = 8 = e = q
    assert t["ep"] == 4 * ring_gather(n, V, alpha, beta)
    assert t["tau"] == t["ep"] / n


def test_expert_parallel_needs_moe_layer():
    inst = make(a2a=10, moe=0, strat=((1, 1, 2, 0, 0),))
    assert O.terms(inst, 0, 1, 1, 0)["valid"] == 0
    assert O.cost_tensor(inst)[0, 1, 0] == O.INF


def test_expert_state_sharded_over_expert_data_parallel_group():
    # 8 devices, EP 4 -> 2 expert replicas; ZeRO-1 shards optimizer state over them
    Pe, opt = 4 * 10**6, 6
    inst = make(pe=Pe, moe=1, opt=opt, strat=((1, 1, 4, 1, 0),))
    t = O.terms(inst, 0, 1, 3, 0)
    We = Pe // 4
    assert t["w"] == We and t["g"] == We and t["o"] == opt * We // 2


def test_context_parallel_gathers():
    n, A, alpha, beta = 4, 8 * 10**6, 100, 10**6
    inst = make(ao=A, G=(8,), bw=(beta,), lat=(alpha,), strat=((1, 4, 1, 0, 0),))
    t = O.terms(inst, 0, 1, 2, 0)
    assert t["cpc"] == 4 * ring_gather(n, A, alpha, beta)


def test_link_cost_is_point_to_point_transfer():
    A = 3 * 10**6
    inst = make(L=3, ao=(A, 2 * A, 5), G=(4, 16), bw=(10**6, 5 * 10**5), lat=(900, 4000),
                cand=(0, 1), D=16)
    X = O.links(inst)
    assert X[0].tolist() == [0, 0] and X[3].tolist() == [0, 0]
    assert X[1].tolist() == [900 + A * 1000 // 10**6, 4000 + A * 1000 // (5 * 10**5)]
    assert X[2].tolist() == [900 + 2 * A * 1000 // 10**6, 4000 + 2 * A * 1000 // (5 * 10**5)]


def test_stash_follows_position_from_pipeline_end():
    """Mem(S, p) = static + (p - 1) stash <= budget, scanned against pmax."""
    rng = np.random.default_rng(5)
    for trial in range(300):
        L = int(rng.integers(1, 5))
        inst = make(L=L, fl=1, pd=rng.integers(0, 10**6, L), ao=rng.integers(0, 10**5, L),
                    aw=rng.integers(0, 10**6, L), Pmax=int(rng.integers(1, 20)),
                    M=64, budget=int(rng.integers(0, 4 * 10**7)),
                    strat=((1, 1, 1, 0, 0), (1, 1, 1, 0, 1), (2, 1, 1, 1, 1)), D=8)
        i = int(rng.integers(0, L))
        j = int(rng.integers(i + 1, L + 1))
        for m in range(4):
            for s in range(3):
                t = O.terms(inst, i, j, m, s)
                if not t["valid"]:
                    continue
                fits = [p for p in range(1, inst.Pmax + 1)
                        if t["stat"] + (p - 1) * t["stash"] <= inst.budget]
                assert t["pmax"] == (max(fits) if fits else 0)
                tc = int(inst.strat[s][0]) * int(inst.strat[s][1])
                if inst.strat[s][4]:   # recompute: only the stage input is stashed
                    ain = int(inst.ao[i - 1]) if i > 0 else int(inst.ao[0])
                    assert t["stash"] == -(-ain // tc)
                    assert t["act"] == -(-int(inst.aw[i:j].max()) // tc)
                else:
                    assert t["stash"] == -(-int(inst.aw[i:j].sum()) // tc)


def _all_terms(inst):
    out = {}
    K = (inst.D // inst.unit).bit_length()
    for i in range(inst.L):
        for j in range(i + 1, inst.L + 1):
            for m in range(K):
                for s in range(inst.S):
                    out[(i, j, m, s)] = O.terms(inst, i, j, m, s)
    return out


@pytest.mark.parametrize("seed", range(12))
def test_monotone_in_rates_latency_and_budget(seed):
    inst = synth.random_tiny(seed + 300, Lmax=4, Dmax=8)
    base = _all_terms(inst)

    faster = synth.random_tiny(seed + 300, Lmax=4, Dmax=8)
    faster.R = inst.R * 2
    faster.tierBw = inst.tierBw * 3
    faster.tierLat = inst.tierLat // 2
    richer = synth.random_tiny(seed + 300, Lmax=4, Dmax=8)
    richer.budget = inst.budget * 2 + 1
    f, r = _all_terms(faster), _all_terms(richer)
    for key, t in base.items():
        if not t["valid"]:
            assert not f[key]["valid"]
            continue
        assert f[key]["tau"] <= t["tau"]
        assert r[key]["pmax"] >= t["pmax"]


def test_zero_stages_never_add_memory():
    rng = np.random.default_rng(11)
    for trial in range(50):
        strat = tuple((2, 1, 2, z, r) for r in (0, 1) for z in range(4))
        inst = make(L=2, pd=rng.integers(0, 10**6, 2), pe=rng.integers(0, 10**6, 2), moe=1,
                    aw=rng.integers(0, 10**5, 2), ao=rng.integers(0, 10**5, 2), strat=strat)
        for m in (1, 2, 3):
            for r in (0, 1):
                st = [O.terms(inst, 0, 2, m, 4 * r + z)["stat"] for z in range(4)]
                assert st[0] >= st[1] >= st[2] >= st[3]


def test_validity_rules():
    strat = ((2, 2, 1, 0, 0), (1, 1, 4, 0, 0), (8, 1, 1, 0, 0))
    inst = make(L=1, moe=1, strat=strat, D=8)
    w = O.cost_tensor(inst)   # [1 pair][4 widths][3 strategies]
    assert (w[0, :2, 0] == O.INF).all() and (w[0, 2:, 0] != O.INF).all()   # t cp | k
    assert (w[0, :2, 1] == O.INF).all() and (w[0, 2:, 1] != O.INF).all()   # e | q
    assert (w[0, :3, 2] == O.INF).all() and w[0, 3, 2] != O.INF            # t | k


@pytest.mark.parametrize("field,value", [
    ("D", 12), ("unit", 3), ("Pmax", 0), ("Pmax", 32), ("M", 1), ("R", 0), ("budget", -1),
    ("opt_factor", 17),
])
def test_invalid_scalars_rejected(field, value):
    inst = synth.config_instance(1, 0)
    setattr(inst, field, value)
    assert O.validate(inst) == 2
    assert O.solve(inst)["status"] == 2


def test_invalid_tables_rejected():
    bad = []
    i = synth.config_instance(2, 0); i.tierG = np.asarray([8, 8, 64]); bad.append(i)
    i = synth.config_instance(2, 0); i.tierG = np.asarray([8, 32, 48]); bad.append(i)
    i = synth.config_instance(2, 0); i.tierG = np.asarray([8, 16, 32]); bad.append(i)   # top < D
    i = synth.config_instance(2, 0); i.tierBw = np.asarray([999, 50000, 25000]); bad.append(i)
    i = synth.config_instance(2, 0); i.cand = np.asarray([2, 0], np.int32); bad.append(i)
    i = synth.config_instance(2, 0); i.strat = i.strat.copy(); i.strat[3, 0] = 3; bad.append(i)
    i = synth.config_instance(2, 0); i.fl = i.fl.copy(); i.fl[5] = (1 << 48) + 1; bad.append(i)
    i = synth.config_instance(2, 0); i.ao = i.ao.copy(); i.ao[0] = (1 << 38) + 1; bad.append(i)
    i = synth.config_instance(2, 0); i.moe = i.moe.copy(); i.moe[0] = 2; bad.append(i)
    for inst in bad:
        assert O.validate(inst) == 2
    assert O.validate(synth.config_instance(2, 0)) == 0


def test_standard_workloads_are_valid():
    for cfg in (1, 2, 3, 4, 5):
        for b in (0, 1):
            if b < synth.CONFIG_BATCH[cfg]:
                assert O.validate(synth.config_instance(cfg, b)) == 0


# ---- expert-parallel gradient sync and ZeRO-3 gathers, and the tiers of groups that
# ---- sit inside a tensor-parallel group.  Two or three tiers with different links make
# ---- the tier choice visible; a wrong group size (q instead of q / e) or tier changes
# ---- every value below.

EXP_TIERS = dict(G=(4, 8), bw=(10**7, 2 * 10**6), lat=(10, 700))   # tier(8) = 1: alpha 700, beta 2e6


def test_expert_gradient_sync_over_the_expert_data_parallel_group():
    # 8 devices, EP 2: the expert weights are data parallel over q / e = 4 replicas, and
    # their gradients are synchronised within that group, on the tier of the whole stage
    Pe = 16 * 10**6
    strat = tuple((1, 1, 2, z, 0) for z in range(4))
    inst = make(pe=Pe, moe=1, M=1, strat=strat, **EXP_TIERS)
    n, We, alpha, beta = 4, Pe // 2, 700, 2 * 10**6
    se = [O.terms(inst, 0, 1, 3, z)["se"] for z in range(4)]
    assert se[0] == ring_allreduce(n, We, alpha, beta)        # no ZeRO: AllReduce
    assert se[1] == se[2] == 2 * ring_gather(n, We, alpha, beta)   # ZeRO-1/2: ReduceScatter + AllGather
    assert se[3] == ring_gather(n, We, alpha, beta)            # ZeRO-3: ReduceScatter only
    # nothing dense to synchronise, and the sync is amortised over the M microbatches
    t0 = O.terms(inst, 0, 1, 3, 0)
    assert t0["sd"] == 0 and t0["tau"] == se[0]


def test_expert_zero3_gathers_over_the_expert_data_parallel_group():
    # ZeRO-3 gathers the expert shards (We / (q / e) each) before the forward and the
    # backward pass of every MoE layer; the dense weights are gathered over all q replicas
    Pd, Pe = 8 * 10**6, 16 * 10**6
    inst = make(pd=Pd, pe=Pe, moe=1, M=1, strat=((1, 1, 2, 3, 0),), **EXP_TIERS)
    q, qe, alpha, beta = 8, 4, 700, 2 * 10**6
    Wd, We = Pd, Pe // 2
    t = O.terms(inst, 0, 1, 3, 0)
    dense = 2 * (q - 1) * alpha + F(q - 1, q) * 2 * Wd * 1000 / beta
    expert = 2 * (qe - 1) * alpha + F(qe - 1, qe) * 2 * We * 1000 / beta
    assert t["z3"] == dense + expert
    assert t["sd"] == ring_gather(q, Wd, alpha, beta) and t["se"] == ring_gather(qe, We, alpha, beta)
    assert t["tau"] == -(-t["z3"] // q) + t["sd"] + t["se"]
    # ZeRO-3 memory: every shard over its own group
    assert t["w"] == Wd // q + We // qe


def test_context_parallel_priced_on_the_tier_of_tp_times_cp():
    # TP 2 x CP 2: the CP pairs are inside a 4-device TP x CP group, so their gathers use
    # the tier that holds 4 devices (tier 1), not the 2-device tier (tier 0) that TP uses
    A = 8 * 10**6
    tiers = dict(G=(2, 4, 8), bw=(8 * 10**6, 2 * 10**6, 10**6), lat=(10, 300, 5000))
    inst = make(ao=A, strat=((2, 2, 1, 0, 0),), **tiers)
    t = O.terms(inst, 0, 1, 2, 0)   # k = 4 = t cp, q = 1
    assert t["cpc"] == 4 * ring_gather(2, A // 2, 300, 2 * 10**6)      # volume Ao / t per collective
    assert t["tp"] == 4 * ring_allreduce(2, A // 2, 10, 8 * 10**6)     # volume Ao / cp per collective
    assert t["tau"] == t["cpc"] + t["tp"]


def test_expert_parallel_priced_on_the_tier_of_tp_times_cp_times_ep():
    # TP 2 x EP 2 on 8 devices: each AllToAll group of 2 lies inside a 4-device TP x EP
    # block, priced on the tier that holds 4 devices; the volume is split over t cp
    V = 16 * 10**6
    tiers = dict(G=(2, 4, 8), bw=(8 * 10**6, 2 * 10**6, 10**6), lat=(10, 300, 5000))
    inst = make(a2a=V, moe=1, strat=((2, 1, 2, 0, 0),), **tiers)
    t = O.terms(inst, 0, 1, 3, 0)   # k = 8, q = 4, q / e = 2
    assert t["ep"] == 4 * ring_gather(2, V // 2, 300, 2 * 10**6)
    assert t["tau"] == t["ep"] / 4


def test_context_and_expert_groups_together():
    # TP 1 x CP 2 x EP 2: CP on tier(2) = 0, EP on tier(4) = 1; with TP 2 both move up
    A, V = 8 * 10**6, 16 * 10**6
    tiers = dict(G=(2, 4, 8), bw=(8 * 10**6, 2 * 10**6, 10**6), lat=(10, 300, 5000))
    inst = make(ao=A, a2a=V, moe=1, strat=((1, 2, 2, 0, 0), (2, 2, 2, 0, 0)), **tiers)
    a = O.terms(inst, 0, 1, 3, 0)   # k = 8: q = 4
    assert a["cpc"] == 4 * ring_gather(2, A, 10, 8 * 10**6)
    assert a["ep"] == 4 * ring_gather(2, V // 2, 300, 2 * 10**6)
    b = O.terms(inst, 0, 1, 3, 1)   # k = 8: t cp = 4, q = 2, e = 2
    assert b["cpc"] == 4 * ring_gather(2, A // 2, 300, 2 * 10**6)
    assert b["ep"] == 4 * ring_gather(2, V // 4, 5000, 10**6)


def test_peak_memory_is_the_sum_of_its_parts():
    """Nest §3.3: Mem(S, p) = 2 weights + optimizer states + activations + (p - 1)
    stashed microbatches.  One layer on k = 2 devices with t = 2 (so q = 1, no ZeRO
    sharding): every part is halved by the tensor split.  The budget is set to the
    p-th position's total and one byte below it, so pmax must be p and p - 1."""
    P, A, f, t = 8 * 10**6, 3 * 10**6, 6, 2
    for p in range(1, 7):
        total = (2 + f) * P // t + A // t + (p - 1) * (A // t)
        for budget, want in ((total, p), (total - 1, p - 1)):
            inst = make(pd=P, aw=A, opt=f, strat=((t, 1, 1, 0, 0),), D=2, G=(2,),
                        Pmax=8, M=8, budget=budget)
            assert O.terms(inst, 0, 1, 1, 0)["pmax"] == want, (p, budget)


def test_peak_memory_with_recompute():
    """With activation recompute a stage keeps one layer's activations at a time (the
    largest) and stashes only its input (the output of the layer before it): stage
    [1, 3) of a three-layer chain, t = 2 on two devices."""
    Pd, aw, ao, f, t = (2 * 10**6, 6 * 10**6, 4 * 10**6), (2 * 10**6, 5 * 10**6, 9 * 10**6), \
        (7 * 10**6, 10**6, 3 * 10**6), 6, 2
    for p in range(1, 7):
        total = (2 + f) * (Pd[1] + Pd[2]) // t + max(aw[1], aw[2]) // t + (p - 1) * (ao[0] // t)
        for budget, want in ((total, p), (total - 1, p - 1)):
            inst = make(L=3, pd=Pd, aw=aw, ao=ao, opt=f, strat=((t, 1, 1, 0, 1),), D=2,
                        G=(2,), Pmax=8, M=8, budget=budget)
            assert O.terms(inst, 1, 3, 1, 0)["pmax"] == want, (p, budget)


def test_context_parallel_splits_compute_and_activations():
    """Context parallelism splits the sequence over its cp devices: each computes a
    cp-th of the layer's flops and holds a cp-th of its activations and stash
    (Nest §3.1 context parallelism; §3.3 memory).  One layer, t = 1, cp = 4 on four
    devices (q = 1), no activation traffic, so no CP collective."""
    F_, A, cp = 4 * 10**6, 8 * 10**6, 4
    strat = ((1, cp, 1, 0, 0),)
    inst = make(fl=F_, aw=A, strat=strat, D=4, G=(4,))
    t = O.terms(inst, 0, 1, 2, 0)
    assert t["comp"] == 3 * F_ // cp and t["cpc"] == 0 and t["tau"] == t["comp"]
    for p in range(1, 6):
        total = A // cp + (p - 1) * (A // cp)
        for budget, want in ((total, p), (total - 1, p - 1)):
            inst = make(fl=F_, aw=A, strat=strat, D=4, G=(4,), Pmax=8, M=8, budget=budget)
            assert O.terms(inst, 0, 1, 2, 0)["pmax"] == want, (p, budget)


def test_expert_alltoall_counts_moe_layers_only():
    """The dispatch and combine AllToAlls are issued by the MoE layers alone: a stage of
    one dense and one MoE layer pays the latency steps of one MoE layer (GShard)."""
    n, V, alpha, beta = 8, 16 * 10**6, 200, 4 * 10**6
    inst = make(L=2, a2a=(0, V), moe=(0, 1), G=(8,), bw=(beta,), lat=(alpha,), strat=((1, 1, 8, 0, 0),))
    t = O.terms(inst, 0, 2, 3, 0)
    assert t["ep"] == 4 * ring_gather(n, V, alpha, beta)
