"""GPU parity of the layered DP sweep (one launch per pipeline position and tag mode,
32-bit tagged words) against the CPU oracle, bit for bit: every DP key, the
per-position loads, the stage-cost words and the results, on every workload, random
tiny instances, layer DAGs, edge cases, and batches that mix instances on rank tags,
on width tags, and instances left to the 64-bit streaming sweep (values beyond the
words).  Nest §4 Eq. 3 is layered in the stage count: position p reads only position
p - 1."""
import numpy as np
import pytest

import gpu_util as G
from memory_aware_device_gb300 import nest, synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu
LAYERED = 3


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


def check_batch(insts, tables=(), chunk=0, keep_costs=True):
    """All results against the oracle; the tables of instances `tables` (indices within
    the last chunk: the workspace holds the last chunk's tables)."""
    s, res = G.run(insts, variant=LAYERED, chunk=chunk, keep_costs=keep_costs)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    first = (len(insts) - 1) // chunk * chunk if chunk else 0
    for b in tables:
        check_tables(s, b - first, insts[b])
    return s, res


def test_layered_launch_description():
    dims = nest.make_dims(synth.config_batch(5, B=4))
    d = nest.describe_launch(dims, nest.options(variant=LAYERED))
    assert d["sweep_variant"] == LAYERED
    # prep, stage loads, position 1, two launches (tag modes) for each of positions
    # 2 .. 16, the streaming launch, backtrack
    assert d["kernels_per_chunk"] == 2 + 1 + 2 * 15 + 1 + 1


def test_layered_workload1():
    inst = synth.config_instance(1, 0)
    assert G.layered_fits(inst)
    check_batch([inst], tables=(0,))


def test_layered_workload2():
    insts = synth.config_batch(2)
    assert all(G.layered_words(x)[0] == 0 and G.layered_fits(x) for x in insts)
    check_batch(insts, tables=(0, 7, 15))


def test_layered_workload3():
    # the deep dense workload's values need 29 bits: width tags
    insts = synth.config_batch(3, B=8)
    assert G.layered_words(insts[0])[0] == 1
    check_batch(insts, tables=(0, 5))


def test_layered_workload4():
    insts = synth.config_batch(4, B=24)
    check_batch(insts, tables=(0, 23))


def test_layered_workload5_tables():
    # instance 2 has the largest values of the first instances (its value bound ~2^26.4)
    insts = synth.config_batch(5, B=3)
    assert all(G.layered_words(x)[0] == 0 and G.layered_fits(x) for x in insts)
    check_batch(insts, tables=(0, 2))


@pytest.mark.parametrize("part", range(3))
def test_layered_random_tiny(part):
    insts = [synth.random_tiny(5000 * part + k, Lmax=7, Dmax=16) for k in range(300)]
    s, res = G.run(insts, Pcap=6, variant=LAYERED)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in range(0, 300, 37):
        if oracle[b]["status"] != 2:
            check_tables(s, b, insts[b])


def test_layered_modes_and_streaming_in_one_solve():
    # flops scaled so that the value bounds spread over rank tags, width tags and beyond
    # the words (those instances saturate and take the 64-bit streaming launch of the
    # same solve)
    base = synth.config_batch(2, B=6)
    factors = (1, 3, 6, 12, 40, 200)
    insts = [G.scaled(x, f) for x, f in zip(base, factors)]
    modes = [G.layered_words(x)[0] for x in insts]
    fits = [G.layered_fits(x) for x in insts]
    assert 0 in modes and 1 in modes and not all(fits), (modes, fits)
    check_batch(insts, tables=range(len(insts)))


def test_layered_values_at_the_word_limits():
    # value bounds just below and above the largest exact value of the rank tags, and
    # just below and above that of the width tags
    x = synth.config_instance(2, 3)
    vb = G.value_bound(x)
    _, tr, vr = G.layered_words(x)
    insts = [G.scaled(x, max(1, int(vr * 0.97) // vb)), G.scaled(x, vr // vb + 1)]
    _, tw, vw = G.layered_words(insts[1])
    insts += [G.scaled(x, max(1, int(vw * 0.97) // vb)), G.scaled(x, vw // vb + 1)]
    modes = [G.layered_words(y)[0] for y in insts]
    fits = [G.layered_fits(y) for y in insts]
    assert modes == [0, 1, 1, 1] and fits == [True, True, True, False], (modes, fits)
    check_batch(insts, tables=range(4))


@pytest.mark.parametrize("part", range(2))
def test_layered_width_tags_random_tiny(part):
    # flops scaled by 2^12: most tiny instances leave the rank tags
    insts = [G.scaled(synth.random_tiny(9000 * part + k, Lmax=7, Dmax=16), 1 << 12) for k in range(300)]
    assert sum(G.layered_words(x)[0] == 1 for x in insts) > 50
    s, res = G.run(insts, Pcap=6, variant=LAYERED)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
    for b in range(0, 300, 41):
        if oracle[b]["status"] != 2:
            check_tables(s, b, insts[b])


def test_layered_graphs():
    insts = [synth.two_tower_instance(0)]
    for k in range(40):
        x = synth.random_tiny(7000 + k, Lmax=7, Dmax=16)
        x.succ = synth.random_dag(k, x.L, (0.0, 0.3, 0.6)[k % 3])
        insts.append(x)
    s, res = G.run(insts, Pcap=16, variant=LAYERED)
    for b, x in enumerate(insts):
        o = G.solve_graph(x)
        assert G.same_graph_result(res[b], o), (b, res[b], o)
    for b in (0, 5, 17):
        G.check_graph_tables(s, b, insts[b])


def test_layered_edge_cases():
    one_layer = synth.config_instance(1, 0)
    one_layer.L = 1
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(one_layer, f, getattr(one_layer, f)[:1])
    p1 = synth.config_instance(2, 1)
    p1.Pmax = 1
    unit = synth.config_instance(2, 2)
    unit.D = unit.unit = 8
    unit.tierG = np.asarray([8, 32, 64])
    zero = synth.config_instance(2, 4)
    zero.budget = 0
    insts = [one_layer, p1, unit, zero, synth.config_instance(2, 5)]
    s, res = G.run(insts, variant=LAYERED)
    oracle = G.oracle_many(insts)
    for b in range(len(insts)):
        assert G.same_result(res[b], oracle[b]), (b, res[b], oracle[b])
        check_tables(s, b, insts[b])
    assert res[3]["status"] == nest.INFEASIBLE


def test_layered_chunks():
    insts = synth.config_batch(4, B=11)
    check_batch(insts, tables=(10,), chunk=4)
