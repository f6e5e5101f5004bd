"""GPU parity for graph instances: Eq. 3 over the up-sets of a layer DAG.

Nest (Network- and Memory-Aware Device Placement) §4 states the DP over downsets of
the operator graph.  The CUDA path enumerates the up-sets in its prep kernel and runs
the same stage-load, sweep and backtrack kernels over pairs of states; every table
and result is compared bit for bit with the oracle's up-set DP.
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


def tiny_graphs(first, n, Lmax=7, Dmax=16):
    out = []
    for k in range(first, first + n):
        x = synth.random_tiny(k, Lmax=Lmax, Dmax=Dmax)
        x.succ = synth.random_dag(k, x.L, (0.0, 0.2, 0.45, 0.8)[k % 4])
        out.append(x)
    return out


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_chain_as_graph_equals_chain_mode(variant):
    chains = synth.config_batch(2, B=4)
    graphs = synth.config_batch(2, B=4)
    for x in graphs:
        x.succ = synth.chain_succ(x.L)
    sc, rc = G.run(chains, variant=variant)
    sg, rg = G.run(graphs, variant=variant)
    for b in range(4):
        o = O.solve(chains[b])
        assert G.same_result(rc[b], o) and G.same_result(rg[b], o), b
        assert rg[b]["layers"] == [((1 << j) - 1) & ~((1 << i) - 1) for i, j, *_ in o["plan"]]
        np.testing.assert_array_equal(G.dp_keys(sg, b, graphs[b]), G.dp_keys(sc, b, chains[b]))
        np.testing.assert_array_equal(G.loads_table(sg, b, graphs[b]), G.loads_table(sc, b, chains[b]))


@pytest.mark.parametrize("part", range(2))
def test_random_dags_match_the_oracle(part):
    insts = tiny_graphs(20000 + 200 * part, 200)
    s, res = G.run(insts)
    oracle = G.oracle_many(insts, fn=G.solve_graph)
    assert sum(o["status"] == 0 for o in oracle) >= 20
    for b in range(len(insts)):
        assert G.same_graph_result(res[b], oracle[b]), b
    for b in range(0, len(insts), 25):
        G.check_graph_tables(s, b, insts[b])


@pytest.mark.parametrize("cluster,jsplit,variant", [(0, 0, 1), (0, 0, 2), (2, 2, 1), (4, 1, 2)])
def test_random_dags_every_table(cluster, jsplit, variant):
    insts = tiny_graphs(21000, 24, Lmax=6, Dmax=8)
    for x in insts:
        x.Pmax = min(x.Pmax, 4)
        x.M = max(x.M, x.Pmax)
    s, res = G.run(insts, cluster=cluster, jsplit=jsplit, variant=variant, Pcap=4)
    for b in range(len(insts)):
        o = G.check_graph_tables(s, b, insts[b])
        assert G.same_graph_result(res[b], o), b


TWO_TOWER_CONFIGS = [(0, 0, 0), (16, 8, 1), (16, 4, 1), (16, 2, 1), (16, 1, 1), (8, 2, 2), (4, 4, 2), (0, 0, 2)]


def test_two_tower_resident_needs_one_position_per_cta():
    # 97 states: the rows of two positions per CTA do not fit in shared memory
    insts = [synth.two_tower_instance(b) for b in range(2)]
    with pytest.raises(nest.NestError) as e:
        G.run(insts, cluster=8, jsplit=4, variant=1)
    assert e.value.rc == nest.NEST_E_LIMITS


@pytest.mark.parametrize("cluster,jsplit,variant", TWO_TOWER_CONFIGS)
def test_two_tower_workload(cluster, jsplit, variant):
    insts = [synth.two_tower_instance(b) for b in range(16)]
    s, res = G.run(insts, cluster=cluster, jsplit=jsplit, variant=variant)
    oracle = G.oracle_many(insts, fn=G.solve_graph)
    assert all(o["status"] == 0 for o in oracle[:4])
    for b in range(len(insts)):
        assert G.same_graph_result(res[b], oracle[b]), b
    for b in (0, 9):
        G.check_graph_tables(s, b, insts[b])


@pytest.mark.parametrize("variant", [1, 2])
def test_two_tower_wide_words(variant):
    insts = [G.scaled(synth.two_tower_instance(b), 64) for b in range(3)]
    s, res = G.run(insts, variant=variant)
    for b in range(len(insts)):
        o = G.check_graph_tables(s, b, insts[b])
        assert G.same_graph_result(res[b], o), b


def test_two_tower_word_kinds():
    # graphs take packed 32-bit words or 64-bit words: values past 2^29 leave no room
    # for the width tag, and plain 32-bit words are not instantiated for graphs.  The
    # chain next to them takes plain 32-bit words at the same values (the width of each
    # best found again at the end of a step)
    chain = G.scaled(synth.config_instance(2, 1), 8)
    insts = [synth.two_tower_instance(0), G.scaled(synth.two_tower_instance(1), 10),
             G.scaled(synth.two_tower_instance(2), 64), chain]
    tb = G.word_tag_bits(insts)
    assert tb == 3
    assert [G.packed_words(x, tb) for x in insts] == [True, False, False, False]
    assert [G.narrow_words(x, tb) for x in insts] == [True, False, False, True]
    for variant in (0, 1):
        s, res = G.run(insts, variant=variant)
        for b in range(3):
            o = G.check_graph_tables(s, b, insts[b])
            assert G.same_graph_result(res[b], o), (variant, b)
        o = O.solve(chain, want_dp=True)
        assert G.same_result(res[3], o), variant
        np.testing.assert_array_equal(G.dp_keys(s, 3, chain), G.oracle_dp_keys(chain, o["dp"]))


def test_chains_and_graphs_in_one_launch():
    insts = synth.config_batch(2, B=3) + [synth.two_tower_instance(b) for b in range(3)]
    insts[1].succ = synth.chain_succ(insts[1].L)
    s, res = G.run(insts)
    for b, x in enumerate(insts):
        o = O.solve(x) if x.succ is None else G.solve_graph(x)
        assert G.same_result(res[b], o), b
    for b in (0, 4):
        if insts[b].succ is None:
            np.testing.assert_array_equal(G.dp_keys(s, b, insts[b]),
                                          G.oracle_dp_keys(insts[b], O.solve(insts[b], want_dp=True)["dp"]))
        else:
            G.check_graph_tables(s, b, insts[b])


def test_bad_graphs_are_flagged_per_instance():
    good = tiny_graphs(22000, 1, Lmax=5)[0]
    back = tiny_graphs(22001, 1, Lmax=5)[0]
    back.L = 5
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(back, f, np.resize(getattr(back, f), 5))
    back.succ = synth.chain_succ(5)
    back.succ[3] |= np.uint64(1 << 1)                     # an edge 3 -> 1
    beyond = tiny_graphs(22002, 1, Lmax=5)[0]
    beyond.succ = synth.chain_succ(beyond.L)
    beyond.succ[0] |= np.uint64(1 << beyond.L)            # an edge to a layer that does not exist
    wide = synth.config_instance(1, 0)                     # 8 independent layers: 256 up-sets
    wide.succ = np.zeros(8, np.uint64)
    long = synth.config_instance(2, 0)                     # a graph of 64 layers
    long.L = 64
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(long, f, np.resize(getattr(long, f), 64))
    long.succ = synth.chain_succ(64)
    insts = [good, back, beyond, wide, long]
    s, res = G.run(insts, Vmax=200)
    assert [r["status"] for r in res[1:]] == [nest.BAD_INPUT] * 4
    assert G.same_graph_result(res[0], G.solve_graph(good))
    # with room for its 255 non-empty up-sets the independent-layer graph solves
    s, res = G.run([wide], Vmax=255, keep_costs=False)
    assert G.same_graph_result(res[0], G.solve_graph(wide))


def test_split_sweep_with_both_word_widths():
    # 16 two-tower instances need two waves when shared memory is sized for 64-bit
    # rows; the sweep then runs as a 32-bit launch and a 64-bit launch, each taking
    # its own instances
    insts = [synth.two_tower_instance(b) for b in range(16)]
    for b in (2, 5, 11):
        insts[b] = G.scaled(insts[b], 64)
    plan = nest.describe_launch(nest.make_dims(insts))
    # prep, stage loads and the two sweep launches; both are resident, so their clusters
    # write the plans and no backtrack kernel runs
    assert plan["sweep_split"] == 1 and plan["kernels_per_chunk"] == 4, plan
    s, res = G.run(insts)
    oracle = G.oracle_many(insts, fn=G.solve_graph)
    for b in range(len(insts)):
        assert G.same_graph_result(res[b], oracle[b]), b
    for b in (2, 3):
        G.check_graph_tables(s, b, insts[b])


def test_widest_graph_matches_chain_mode():
    # 63 layers as a graph (bit 62 of the masks in use) against the same chain
    base = synth.config_instance(2, 5)
    base.L, base.Pmax = 63, 8
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(base, f, np.resize(getattr(base, f), 63))
    import copy
    g = copy.deepcopy(base)
    g.succ = synth.chain_succ(63)
    s, res = G.run([base, g])
    o = O.solve(base, want_dp=True)
    assert G.same_result(res[0], o) and G.same_result(res[1], o)
    assert res[1]["layers"][0] & (1 << 62) or res[1]["layers"][-1] & (1 << 62)
    np.testing.assert_array_equal(G.dp_keys(s, 1, g), G.oracle_dp_keys(base, o["dp"]))


def test_largest_state_count_on_the_dense_tiers():
    # 8 independent layers (every subset is an up-set: 256 states, the most the 8-bit
    # state index allows) with the dense workload's tiers, widths and strategies, next
    # to a chain instance in the same batch
    g = synth.config_instance(2, 2)
    g.L, g.Pmax, g.M = 8, 8, 64
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(g, f, np.resize(getattr(g, f), 8))
    g.succ = np.zeros(8, np.uint64)
    chain = synth.config_instance(2, 3)
    chain.Pmax = 8
    s, res = G.run([g, chain], Vmax=255)
    og = G.check_graph_tables(s, 0, g)
    assert og["status"] == 0 and len(og["states"]) == 256
    assert G.same_graph_result(res[0], og)
    assert G.same_result(res[1], O.solve(chain))


def test_graph_batches_in_ragged_chunks():
    # passes of 7 instances over a mix of DAGs and chains give the oracle's results
    insts = tiny_graphs(23000, 40, Lmax=7, Dmax=16)
    for x in insts[::3]:
        x.succ = None
    s, res = G.run(insts, chunk=7, keep_costs=False)
    for b, x in enumerate(insts):
        o = O.solve(x) if x.succ is None else G.solve_graph(x)
        assert G.same_result(res[b], o), b
        if x.succ is not None:
            assert G.same_graph_result(res[b], o), b
