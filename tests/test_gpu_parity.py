"""GPU parity: every kernel of the CUDA path against the CPU oracle, bit for bit.

All quantities are int64 nanoseconds, bytes and packed integer keys, so the bar is
exact equality: the stage-cost words (cost builder), the per-position strategy
loads (reduction), every DP cell key (sweep), and the batch time, bottleneck and
plan (backtrack).  Workloads 1, 2 and 4 are compared in full; workload 3 on its
full batch with every result checked and two instances' tables checked cell by
cell; workload 5 at its full size (1024 instances, chunked) on every result, against
the oracle's stored results, and two instances' tables.
"""
import numpy as np
import pytest

import gpu_util as G
from memory_aware_device_gb300 import nest, synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    G.ensure_built()


def check_tables(s, b, inst):
    np.testing.assert_array_equal(G.cost_table(s, b, inst), O.cost_tensor(inst))
    np.testing.assert_array_equal(G.loads_table(s, b, inst), O.loads(inst))
    o = O.solve(inst, want_dp=True)
    np.testing.assert_array_equal(G.dp_keys(s, b, inst), G.oracle_dp_keys(inst, o["dp"]))
    return o


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_workload1_all_tables(variant):
    inst = synth.config_instance(1, 0)
    s, res = G.run([inst], variant=variant)
    o = check_tables(s, 0, inst)
    assert G.same_result(res[0], o)


# (CTAs per instance, threads per cell, sweep variant: 0 auto, 1 resident, 2 streaming)
SWEEP_CONFIGS = [(0, 0, 0), (1, 1, 2), (2, 2, 2), (4, 4, 2), (8, 8, 1), (4, 2, 2), (8, 4, 1), (8, 1, 2),
                 (8, 2, 1), (16, 4, 1), (16, 8, 1), (16, 8, 2), (16, 1, 1), (16, 2, 1)]


def test_resident_variant_rejected_when_it_does_not_fit():
    # 2 CTAs per instance would hold the rows of 8 positions each: about 270 KB per CTA
    insts = synth.config_batch(2, B=2)
    with pytest.raises(nest.NestError) as e:
        G.run(insts, cluster=2, jsplit=4, variant=1)
    assert e.value.rc == nest.NEST_E_LIMITS


def test_resident_variant_needs_a_peer_cta():
    # rows go to the next position's CTA by st.async, which must be another CTA: one
    # CTA per instance is refused before any launch when there is more than one position
    insts = synth.config_batch(2, B=2)
    with pytest.raises(nest.NestError) as e:
        G.run(insts, cluster=1, jsplit=4, variant=1)
    assert e.value.rc == nest.NEST_E_LIMITS


@pytest.mark.parametrize("cluster,jsplit,variant", SWEEP_CONFIGS)
def test_workload2_all_tables(cluster, jsplit, variant):
    insts = synth.config_batch(2)
    s, res = G.run(insts, cluster=cluster, jsplit=jsplit, variant=variant)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    for b in (0, 7, 15):
        check_tables(s, b, insts[b])


# The resident sweep keeps 32-bit value words when every value is small and 64-bit
# words otherwise; flops scaled by 64 push workload 2's loads past 2^30.
@pytest.mark.parametrize("cluster,jsplit,variant", [(0, 0, 1), (16, 8, 1), (8, 4, 1), (8, 2, 1), (16, 1, 1),
                                                    (0, 0, 2)])
def test_workload2_wide_words(cluster, jsplit, variant):
    insts = [G.scaled(x, 64) for x in synth.config_batch(2, B=4)]
    assert not any(G.narrow_words(x) for x in insts)
    s, res = G.run(insts, cluster=cluster, jsplit=jsplit, variant=variant)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
        check_tables(s, b, insts[b])


def test_packed_words_near_their_limit():
    # two candidates and 64 device counts: 32-bit words packed with 3 tag bits, exact for
    # values up to 2^29 - 2.  Flops scaled so that the value bounds lie at 0.71 and 0.91 x
    # 2^29 (packed words, their top value bits in use), at 1.04 and 1.27 x 2^29 (plain
    # 32-bit words: no room for the tag) and beyond 2^30 (64-bit words), all in one launch
    base = synth.config_batch(2, B=5)
    insts = [G.scaled(base[0], 7), G.scaled(base[1], 7), G.scaled(base[2], 7), G.scaled(base[3], 12),
             G.scaled(base[4], 64)]
    tb = G.word_tag_bits(insts)
    assert tb == 3
    assert [G.packed_words(x, tb) for x in insts] == [True, True, False, False, False]
    assert [G.narrow_words(x) for x in insts] == [True, True, True, True, False]
    assert G.value_bound(insts[1]) > 2**28 + 2**27
    for variant in (0, 1):
        s, res = G.run(insts, variant=variant)
        oracle = G.oracle_many(insts)
        for b in range(len(insts)):
            assert G.same_result(res[b], oracle[b]), (variant, b)
            check_tables(s, b, insts[b])


def tagged_batch(n=90):
    """Random instances with one or two link candidates (tagged 32-bit words), flops
    scaled so that the value bounds spread over packed words, plain 32-bit words and
    64-bit words."""
    xs, k = [], 0
    while len(xs) < n:
        x = synth.random_tiny(31000 + k, Lmax=7, Dmax=16)
        k += 1
        if len(x.cand) <= 2 and G.value_bound(x) > 0:
            xs.append(x)
    targets = (0.3, 0.9, 1.3, 1.8, 2.5)   # x 2^29
    return [G.scaled(x, max(1, round(targets[b % 5] * 2**29 / G.value_bound(x)))) for b, x in enumerate(xs)]


@pytest.mark.parametrize("variant", [0, 1])
def test_tagged_words_on_random_instances(variant):
    insts = tagged_batch()
    tb = G.word_tag_bits(insts)
    kind = ["packed" if G.packed_words(x, tb) else "plain" if G.narrow_words(x) else "wide" for x in insts]
    assert tb == 3 and min(kind.count(k) for k in ("packed", "plain", "wide")) >= 5
    s, res = G.run(insts, Pcap=6, variant=variant)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, kind[b])
    for k in ("packed", "plain", "wide"):
        for b in [b for b in range(len(insts)) if kind[b] == k][:4]:
            check_tables(s, b, insts[b])


def test_mixed_word_widths_in_one_launch():
    insts = synth.config_batch(2, B=6)
    for b in (1, 3, 4):
        insts[b] = G.scaled(insts[b], 64)
    assert [G.narrow_words(x) for x in insts] == [True, False, True, False, False, True]
    s, res = G.run(insts, variant=1)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
        check_tables(s, b, insts[b])


# GPipe stash schedule: memory at every position as for all ceil(M / q) microbatches
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_workload2_gpipe_all_tables(variant):
    insts = synth.config_batch(2, B=8)
    for x in insts:
        x.schedule, x.M = 1, 512
    s, res = G.run(insts, variant=variant)
    oracle = G.oracle_many(insts)
    assert sum(o["status"] == 0 for o in oracle) >= 4
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
        check_tables(s, b, insts[b])


def test_mixed_schedules_in_one_launch():
    insts = [synth.random_tiny(3000 + k, Lmax=7, Dmax=16) for k in range(200)]
    for x in insts[::2]:
        x.schedule = 1
    s, res = G.run(insts, Pcap=6)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    for b in range(0, 200, 23):
        if oracle[b]["status"] != 2:
            check_tables(s, b, insts[b])


# Joint microbatch-size search: each problem's variants are consecutive instances
def _joint_check(problems, **kw):
    import torch
    insts = synth.joint_batch(problems)
    group = len(synth.MICROBATCH_SIZES)
    s, res = G.run(insts, **kw)
    best = nest.select_best(s.costs, group)
    torch.cuda.synchronize()
    best = best.cpu().tolist()
    for g, x in enumerate(problems):
        j = O.solve_joint(insts[g * group:(g + 1) * group])
        for q in range(group):
            assert G.same_result(res[g * group + q], j["results"][q]), (g, q)
        assert best[g] == j["best"], (g, best[g], j["best"])
    return best


def test_joint_microbatch_search_workload2():
    best = _joint_check(synth.config_batch(2, B=6))
    assert len(set(best)) >= 1


def test_joint_microbatch_search_random_tiny():
    best = _joint_check([synth.random_tiny(4000 + k, Lmax=7, Dmax=16) for k in range(60)], Pcap=6)
    assert -1 in best or len(set(best)) > 1   # the sample exercises different answers


# Torus cluster: hop-distance tiers (1-hop pairs, 2-hop squares, the whole torus)
def test_torus_workload_all_tables():
    insts = [synth.torus_instance(b) for b in range(16)]
    s, res = G.run(insts)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    for b in (0, 9, 15):
        check_tables(s, b, insts[b])


def test_workload3_full_batch():
    insts = synth.config_batch(3)
    s, res = G.run(insts)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    for b in (0, 63):
        check_tables(s, b, insts[b])


def test_workload4_full_batch():
    insts = synth.config_batch(4)
    s, res = G.run(insts)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    for b in (0, 100, 255):
        check_tables(s, b, insts[b])


def _golden5():
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "make_workload5_results.py")
    spec = importlib.util.spec_from_file_location("make_workload5_results", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def workload5():
    """The 1024 instances of the mixed-128L workload, the oracle's stored results for
    them (tests/golden/workload5_results.txt, written by the oracle alone), and the
    oracle's tables of two instances of the last chunk of 152."""
    mod = _golden5()
    insts = synth.config_batch(5)
    gold = mod.parse()
    assert sorted(gold) == list(range(1024))
    for b, x in enumerate(insts):   # the generator still draws the inputs the file was written for
        assert gold[b][0] == mod.fingerprint(x), b
    last0 = (1024 // 152) * 152
    tables = {}
    for b in (last0, 1023):
        o = O.solve(insts[b], want_dp=True)
        tables[b] = (O.cost_tensor(insts[b]), O.loads(insts[b]), G.oracle_dp_keys(insts[b], o["dp"]))
    return insts, gold, tables, last0


@pytest.mark.parametrize("variant,keep_costs", [(0, True), (2, True), (0, False)])
def test_workload5_full_size_all_instances(workload5, variant, keep_costs):
    """All 1024 instances solved in chunks of 152 (the library's sweep choice, and the
    streaming variant): every status, t_batch, bottleneck and plan against the oracle's
    stored results, and every table (stage-cost words when kept, per-position loads, DP
    keys) of two instances against the oracle.  Without the kept cost tensor the stage
    loads take the path that never prices strategy groups fitting no position, which is
    the one solves take by default."""
    insts, gold, tables, last0 = workload5
    s, res = G.run(insts, chunk=152, variant=variant, keep_costs=keep_costs)
    for b in range(1024):
        _, st, t, v, plan = gold[b]
        assert (res[b]["status"], res[b]["t_batch"]) == (st, t), (b, res[b])
        if st == 0:
            assert res[b]["bottleneck"] == v and res[b]["plan"] == plan, (b, res[b])
    for b, (cost, loads, keys) in tables.items():
        if keep_costs:
            np.testing.assert_array_equal(G.cost_table(s, b - last0, insts[b]), cost)
        np.testing.assert_array_equal(G.loads_table(s, b - last0, insts[b]), loads)
        np.testing.assert_array_equal(G.dp_keys(s, b - last0, insts[b]), keys)


@pytest.mark.parametrize("cfg,B", [(2, 16), (3, 4), (4, 12)])
def test_loads_without_kept_costs(cfg, B):
    """The stage loads solves take by default (no kept cost tensor: strategy groups that
    fit no position are never priced): results, per-position loads and DP keys against
    the oracle."""
    insts = synth.config_batch(cfg, B=B)
    s, res = G.run(insts, keep_costs=False)
    oracle = G.oracle_many(insts)
    for b in range(B):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in (0, B - 1):
        np.testing.assert_array_equal(G.loads_table(s, b, insts[b]), O.loads(insts[b]))
        o = O.solve(insts[b], want_dp=True)
        np.testing.assert_array_equal(G.dp_keys(s, b, insts[b]), G.oracle_dp_keys(insts[b], o["dp"]))


def test_loads_without_kept_costs_tight_budgets():
    # budgets from generous to an eighth: more and more strategy groups fit no position
    insts = []
    for k in range(240):
        x = synth.random_tiny(52000 + k, Lmax=7, Dmax=16)
        x.budget = int(x.budget) // (1 + k % 8)
        insts.append(x)
    s, res = G.run(insts, Pcap=6, keep_costs=False)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in range(0, 240, 23):
        if oracle[b]["status"] != 2:
            np.testing.assert_array_equal(G.loads_table(s, b, insts[b]), O.loads(insts[b]))


@pytest.mark.parametrize("part,variant,factor", [(0, 0, 1), (1, 1, 1), (2, 2, 1), (3, 1, 1), (4, 1, 1 << 20)])
def test_random_tiny_batches(part, variant, factor):
    insts = [G.scaled(synth.random_tiny(1000 * part + k, Lmax=7, Dmax=16), factor) for k in range(300)]
    if factor > 1:   # most take the 64-bit words of the resident sweep, some the 32-bit ones
        assert 0 < sum(G.narrow_words(x) for x in insts) < 100
    s, res = G.run(insts, Pcap=6, variant=variant)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in range(0, 300, 37):
        if oracle[b]["status"] != 2:
            check_tables(s, b, insts[b])


def test_lowest_bandwidth_tiers():
    # every tier at the smallest allowed bandwidth (1000 bytes/us): every ring transfer's
    # bytes divide exactly, so the rounding cases of the collective prices (shared
    # between the AllReduce and the AllGather of a group) all occur
    insts = []
    for k in range(200):
        x = synth.random_tiny(41000 + k, Lmax=7, Dmax=16)
        x.tierBw = np.full(len(x.tierBw), 1000, dtype=np.int64) + (k % 2) * np.arange(len(x.tierBw))
        insts.append(x)
    s, res = G.run(insts, Pcap=6)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in range(0, 200, 13):
        if oracle[b]["status"] != 2:
            check_tables(s, b, insts[b])


def test_ragged_chunks_and_mixed_shapes():
    """Instances of different sizes in one batch, processed in ragged chunks."""
    insts = synth.config_batch(2, B=5) + synth.config_batch(1) + \
        [synth.random_tiny(k, Lmax=7, Dmax=16) for k in range(11)]
    oracle = G.oracle_many(insts)
    for chunk in (0, 4, 7):
        s, res = G.run(insts, chunk=chunk)
        for b in range(len(insts)):
            assert G.same_result(res[b], oracle[b]), (chunk, b)


def test_edge_cases():
    one_layer = synth.config_instance(1, 0)
    one_layer.L = 1
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(one_layer, f, getattr(one_layer, f)[:1].copy())
    single_stage = synth.config_instance(2, 1)
    single_stage.Pmax = 1
    one_unit = synth.config_instance(4, 0)
    one_unit.D = one_unit.unit
    starved = synth.config_instance(2, 2)
    starved.budget = 0
    bad = synth.config_instance(2, 3)
    bad.tierBw = np.asarray([900000, 999, 25000], np.int64)
    bad2 = synth.config_instance(2, 4)
    bad2.M = 3   # below Pmax
    insts = [one_layer, single_stage, one_unit, starved, bad, bad2, synth.config_instance(2, 5)]
    s, res = G.run(insts)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), b
    assert [r["status"] for r in res][3:6] == [nest.INFEASIBLE, nest.BAD_INPUT, nest.BAD_INPUT]


def test_maximum_positions():
    """Pcap = 31 stages (the largest the keys allow) on a 40-layer chain."""
    inst = synth.config_instance(2, 6)
    L = 40
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        a = getattr(inst, f)
        setattr(inst, f, np.resize(a, L).astype(a.dtype))
    inst.L, inst.Pmax, inst.budget = L, 31, 12 * 10**9
    s, res = G.run([inst])
    o = check_tables(s, 0, inst)
    assert G.same_result(res[0], o)


def test_deterministic_bytes():
    insts = synth.config_batch(2)
    s1, r1 = G.run(insts)
    s2, r2 = G.run(insts)
    assert r1 == r2
    assert (s1.plans.cpu().numpy() == s2.plans.cpu().numpy()).all()


def test_host_entry_point_matches_device_entry_point():
    import torch
    insts = synth.config_batch(2)
    dims = nest.make_dims(insts)
    rec = nest.pack_records(insts, dims)
    ws = torch.empty(nest.workspace_size(dims, host=True), dtype=torch.uint8, device="cuda")
    costs = np.zeros(dims.B, np.int64)
    plans = np.zeros(dims.B * nest.plan_bytes(dims), np.uint8)
    assert nest.solve_host_raw(dims, rec, costs, plans, ws) == nest.NEST_OK
    _, res = G.run(insts)
    assert nest.decode_plans(plans, dims) == res
    assert costs.tolist() == [r["t_batch"] for r in res]


@pytest.mark.parametrize("variant", [1, 2])
def test_bounded_wait_gives_up_and_context_survives(variant):
    """A wait forced to give up marks the instances NEST_TIMED_OUT; the GPU context
    stays usable and the next call is exact again."""
    import torch
    insts = synth.config_batch(2, B=4)
    _, res = G.run(insts, spin_limit=-1, variant=variant)
    assert all(r["status"] == nest.TIMED_OUT and r["t_batch"] == -1 for r in res)
    dims = nest.make_dims(insts)
    ws = torch.empty(nest.workspace_size(dims, host=True), dtype=torch.uint8, device="cuda")
    costs = np.zeros(dims.B, np.int64)
    plans = np.zeros(dims.B * nest.plan_bytes(dims), np.uint8)
    rc = nest.solve_host_raw(dims, nest.pack_records(insts, dims), costs, plans, ws,
                             opt=nest.options(spin_limit=-1))
    assert rc == nest.NEST_E_TIMEOUT
    _, res2 = G.run(insts)
    oracle = G.oracle_many(insts)
    assert all(G.same_result(a, b) for a, b in zip(res2, oracle))


def test_torus_split_sweep_mixed_widths():
    # three candidate tiers: the resident rows of both widths need two waves for 16
    # instances, so the sweep is split by word width
    insts = [synth.torus_instance(b) for b in range(16)]
    for b in (0, 9):
        insts[b] = G.scaled(insts[b], 64)
    plan = nest.describe_launch(nest.make_dims(insts))
    s, res = G.run(insts)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, plan)
    for b in (0, 1):
        check_tables(s, b, insts[b])


@pytest.mark.parametrize("workload", [1, 2])
def test_solve_replays_from_a_cuda_graph(workload):
    # nest_solve only enqueues kernels (no allocation, no synchronisation), so a caller
    # can capture it once and replay it; the replays give the direct results
    import torch
    insts = synth.config_batch(workload)
    dims = nest.make_dims(insts)
    s = nest.Solver(dims)
    s.load(nest.pack_records(insts, dims))
    s.run()
    torch.cuda.synchronize()
    want = s.results()
    graph = s.capture()
    torch.cuda.synchronize()
    for _ in range(2):
        s.plans.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert s.results() == want
