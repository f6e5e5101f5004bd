"""Pins for the oracle's DP over the up-sets of a layer DAG.

Nest (Network- and Memory-Aware Device Placement) §4 states Eq. 3 over downsets of
the operator graph: a state is the set of layers still to be placed, a stage the
difference of two states.  Read here for a topologically numbered DAG: the states
are the up-sets, a transition goes from D to an up-set strictly inside it, and the
bytes entering D (outputs of the layers outside D that feed it; for the whole graph
the source layers' outputs) are the link volume and the stage's stashed input.

Pinned by (1) the states against a scan of every layer subset; (2) the mask stage
terms against the chain terms of the same layers gathered into a chain; (3) the
link costs against their definition computed from the edge list; (4) a chain
written as a DAG reproducing the chain solver's tables and plans bit for bit; (5)
exhaustive enumeration of every plan (chains of up-sets x widths x tiers x
strategies) on tiny DAGs; (6) invariance of the optimum under a different
topological numbering of the same graph; (7) an extra constraint edge never
lowering the optimum.
"""
import dataclasses
import itertools

import numpy as np
import pytest

from memory_aware_device_gb300 import synth
from oracle import oracle as O

CAP = (1 << 40) - 1
INF = (1 << 64) - 1


def edges(succ):
    return [(u, v) for u in range(len(succ)) for v in range(len(succ)) if int(succ[u]) >> v & 1]


def entering(L, succ, D):
    """Bytes-entering set of layers for up-set D, from the edge list."""
    E = edges(succ)
    full = (1 << L) - 1
    if D == full:
        return [l for l in range(L) if not any(v == l for _, v in E)]
    return sorted({u for u, v in E if D >> v & 1 and not D >> u & 1})


def is_upset(succ, D):
    return all(not (D >> u & 1) or (int(succ[u]) & ~D) == 0 for u in range(len(succ)))


def tiny(seed, Lmax=6, **kw):
    x = synth.random_tiny(seed, Lmax=Lmax, **kw)
    dens = (0.0, 0.25, 0.5, 0.8)[seed % 4]
    return x, synth.random_dag(seed, x.L, dens)


@pytest.mark.parametrize("seed", range(40))
def test_states_are_the_upsets(seed):
    L = 1 + seed % 9
    succ = synth.random_dag(seed, L, (0.15, 0.4, 0.7)[seed % 3])
    x = synth.random_tiny(seed)
    x.L = L
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(x, f, np.resize(getattr(x, f), L))
    st = O.lattice_states(x, succ)
    want = [D for D in range(1 << L) if is_upset(succ, D)]
    if len(want) > 256:
        assert st is None
        return
    assert sorted(int(v) for v in st) == want
    key = [(-bin(int(v)).count("1"), int(v)) for v in st]
    assert key == sorted(key)
    assert int(st[0]) == (1 << L) - 1 and int(st[-1]) == 0


def test_state_limits():
    x = synth.random_tiny(2, Lmax=9)
    x.L = 9
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(x, f, np.resize(getattr(x, f), 9))
    assert O.lattice_states(x, np.zeros(9, np.uint64)) is None          # 512 up-sets
    assert O.solve_lattice(x, np.zeros(9, np.uint64))["status"] == 2
    back = synth.chain_succ(9)
    back[3] |= np.uint64(1 << 1)                                         # an edge 3 -> 1
    assert O.lattice_states(x, back) is None
    assert O.solve_lattice(x, back)["status"] == 2


@pytest.mark.parametrize("seed", range(60))
def test_mask_terms_equal_gathered_chain_terms(seed):
    x, succ = tiny(seed, Lmax=7)
    st = [int(v) for v in O.lattice_states(x, succ)]
    rng = np.random.default_rng(seed)
    K = (x.D // x.unit).bit_length()
    for _ in range(6):
        a, b = sorted(rng.choice(len(st), size=2, replace=len(st) < 2))
        if a == b or (st[b] & ~st[a]):
            continue
        D, Dp = st[a], st[b]
        S = [l for l in range(x.L) if (D & ~Dp) >> l & 1]
        ain = sum(int(x.ao[l]) for l in entering(x.L, succ, D))
        # a chain: one producer layer whose output is the bytes entering D, then the
        # stage's layers in order; chain stage [1, 1 + |S|) has the same sums
        y = dataclasses.replace(x)
        y.L = 1 + len(S)
        for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
            v = np.asarray(getattr(x, f))
            setattr(y, f, np.concatenate([np.zeros(1, v.dtype), v[S]]))
        y.ao = y.ao.copy()
        y.ao[0] = ain
        for m in range(K):
            for s in range(len(x.strat)):
                assert O.lattice_terms(x, succ, D, Dp, m, s) == O.terms(y, 1, y.L, m, s)


@pytest.mark.parametrize("seed", range(40))
def test_links_follow_the_edge_list(seed):
    x, succ = tiny(seed, Lmax=7)
    full = (1 << x.L) - 1
    for D in (int(v) for v in O.lattice_states(x, succ)):
        for c in range(len(x.cand)):
            got = O.lattice_link(x, succ, D, c)
            if D in (0, full):
                assert got == 0
                continue
            tr = int(x.cand[c])
            byt = sum(int(x.ao[l]) for l in entering(x.L, succ, D))
            assert got == int(x.tierLat[tr]) + -(-byt * 1000 // int(x.tierBw[tr]))


@pytest.mark.parametrize("seed", range(80))
def test_chain_as_dag_is_the_chain_solver(seed):
    x = synth.random_tiny(seed + 300, Lmax=8, Dmax=16)
    succ = synth.chain_succ(x.L)
    st = O.lattice_states(x, succ)
    assert [int(v) for v in st] == [((1 << x.L) - 1) ^ ((1 << i) - 1) for i in range(x.L + 1)]
    pairs, ld = O.lattice_loads(x, succ)
    assert pairs == [(i, j) for i in range(x.L) for j in range(i + 1, x.L + 1)]
    assert np.array_equal(ld, O.loads(x))
    a, b = O.solve(x, want_dp=True), O.solve_lattice(x, succ, want_dp=True)
    assert (a["status"], a["t_batch"], a["bottleneck"], a["plan"]) == \
        (b["status"], b["t_batch"], b["bottleneck"], b["plan"])
    assert np.array_equal(a["dp"], b["dp"])


def test_chain_as_dag_on_the_dense_workload():
    x = synth.config_instance(2, 3)
    a, b = O.solve(x, want_dp=True), O.solve_lattice(x, synth.chain_succ(x.L), want_dp=True)
    assert a["plan"] == b["plan"] and a["t_batch"] == b["t_batch"]
    assert np.array_equal(a["dp"], b["dp"])


# --- exhaustive enumeration -------------------------------------------------------

def brute_lattice(x, succ):
    """Every plan: a chain of up-sets full = D_0 > D_1 > ... > D_P = {}, a width per
    stage, a candidate tier per internal link; each stage takes the fastest strategy
    that fits its position P - q.  Returns the best (t_batch, P, bottleneck)."""
    L, Du, unit = x.L, x.D // x.unit, x.unit
    K = Du.bit_length()
    G = [int(g) for g in x.tierG]
    cand = [int(c) for c in x.cand]
    C = len(cand)
    full = (1 << L) - 1
    ups = [D for D in range(1 << L) if is_upset(succ, D)]

    words = {}

    def tau_at(D, Dp, m, pos):
        if (D, Dp, m) not in words:
            row = []
            for s in range(len(x.strat)):
                t = O.lattice_terms(x, succ, D, Dp, m, s)
                row.append(None if not t["valid"] or t["tau"] >= CAP else (t["tau"], t["pmax"]))
            words[(D, Dp, m)] = row
        best = None
        for w in words[(D, Dp, m)]:
            if w is not None and w[1] >= pos and (best is None or w[0] < best):
                best = w[0]
        return best

    def link(D, c):
        if D in (0, full):
            return 0
        tr = cand[c]
        byt = sum(int(x.ao[l]) for l in entering(L, succ, D))
        return int(x.tierLat[tr]) + -(-byt * 1000 // int(x.tierBw[tr]))

    def chains(D, n):
        if n == 0:
            if D == 0:
                yield (0,)
            return
        for E in ups:
            if E != D and (E & ~D) == 0:
                for rest in chains(E, n - 1):
                    yield (D,) + rest

    best = None
    for P in range(1, min(x.Pmax, L) + 1):
        for ch in chains(full, P):
            for ms in itertools.product(range(K), repeat=P):
                if sum(1 << m for m in ms) > Du:
                    continue
                taus = [tau_at(ch[q], ch[q + 1], ms[q], P - q) for q in range(P)]
                if any(t is None for t in taus):
                    continue
                for cs in itertools.product(range(C), repeat=P - 1):
                    bott, ok = 0, True
                    for q in range(P):
                        k = unit << ms[q]
                        cost = taus[q]
                        if q > 0:
                            ok &= 2 * k <= G[cand[cs[q - 1]]]
                            cost += link(ch[q], cs[q - 1])
                        if q < P - 1:
                            ok &= 2 * k <= G[cand[cs[q]]]
                            cost += link(ch[q + 1], cs[q])
                        bott = max(bott, cost)
                    if not ok or bott >= CAP:
                        continue
                    t = bott * (x.M + P - 1)
                    if best is None or (t, P) < (best[0], best[1]):
                        best = (t, P, bott)
    return best


@pytest.mark.parametrize("chunk", range(4))
def test_lattice_dp_matches_exhaustive_enumeration(chunk):
    solved = 0
    for seed in range(chunk * 60, (chunk + 1) * 60):
        x, succ = tiny(seed + 9000, Lmax=5, Dmax=4, Cmax=2)
        x.Pmax = min(x.Pmax, 4)
        x.M = max(x.M, x.Pmax)
        b = brute_lattice(x, succ)
        r = O.solve_lattice(x, succ)
        if b is None:
            assert r["status"] == 1
            continue
        assert r["status"] == 0 and (r["t_batch"], len(r["plan"]), r["bottleneck"]) == b, seed
        solved += 1
        # the returned plan is a chain of up-sets covering the graph
        st = [int(v) for v in r["states"]]
        assert r["plan"][0][0] == 0 and r["plan"][-1][1] == len(st) - 1
        for (i, j, k, s, c), nxt in zip(r["plan"], r["plan"][1:] + [None]):
            assert st[j] != st[i] and (st[j] & ~st[i]) == 0
            assert nxt is None or nxt[0] == j
    assert solved > 10


def relabel(x, succ, perm):
    """The same graph with layer l renamed perm[l] (perm a topological order)."""
    y = dataclasses.replace(x)
    inv = np.argsort(perm)
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(y, f, np.asarray(getattr(x, f))[inv])
    out = np.zeros(x.L, np.uint64)
    for u, v in edges(succ):
        out[perm[u]] |= np.uint64(1 << int(perm[v]))
    return y, out


def random_topological_order(succ, rng):
    L = len(succ)
    indeg = [sum(1 for u, v in edges(succ) if v == l) for l in range(L)]
    ready = [l for l in range(L) if indeg[l] == 0]
    perm = [0] * L
    for pos in range(L):
        l = ready.pop(int(rng.integers(len(ready))))
        perm[l] = pos
        for u, v in edges(succ):
            if u == l:
                indeg[v] -= 1
                if indeg[v] == 0:
                    ready.append(v)
    return perm


@pytest.mark.parametrize("seed", range(60))
def test_optimum_is_invariant_under_renumbering(seed):
    x, succ = tiny(seed + 400, Lmax=7, Dmax=16)
    perm = random_topological_order(succ, np.random.default_rng(seed))
    y, sy = relabel(x, succ, perm)
    a, b = O.solve_lattice(x, succ), O.solve_lattice(y, sy)
    assert (a["status"], a["t_batch"], a["bottleneck"], len(a["plan"])) == \
        (b["status"], b["t_batch"], b["bottleneck"], len(b["plan"]))


@pytest.mark.parametrize("seed", range(60))
def test_extra_edge_never_helps(seed):
    # an edge into a layer that already has a producer keeps the sources, removes
    # up-sets and only adds bytes entering a state
    x, succ = tiny(seed + 700, Lmax=7, Dmax=16)
    E = edges(succ)
    rng = np.random.default_rng(seed)
    new = [(u, v) for u in range(x.L) for v in range(u + 1, x.L)
           if (u, v) not in E and any(w == v for _, w in E)]
    if not new:
        return
    u, v = new[int(rng.integers(len(new)))]
    s2 = succ.copy()
    s2[u] |= np.uint64(1 << v)
    a, b = O.solve_lattice(x, succ), O.solve_lattice(x, s2)
    if a["status"] == 1:
        assert b["status"] == 1
    elif b["status"] == 0:
        assert b["t_batch"] >= a["t_batch"]


def test_single_stage_is_the_whole_graph():
    # with one pipeline stage every DAG with a single source gives the chain's answer
    for seed in range(40):
        x, succ = tiny(seed + 1100, Lmax=7)
        x.Pmax = 1
        x.M = max(x.M, 1)
        for v in range(1, x.L):
            succ[0] |= np.uint64(1 << v)           # layer 0 feeds every other layer
        a, b = O.solve(x), O.solve_lattice(x, succ)
        assert (a["status"], a["t_batch"], a["plan"][:1] and a["plan"][0][2:]) == \
            (b["status"], b["t_batch"], b["plan"][:1] and b["plan"][0][2:])


def test_two_tower_workload():
    x, succ = synth.two_tower_instance(0), synth.two_tower_succ()
    st = O.lattice_states(x, succ)
    assert len(st) == 17 + 9 * 9 - 1
    r = O.solve_lattice(x, succ)
    assert r["status"] == 0
    # both branches feed the first stage: its stash is ao[0] + ao[8]
    assert entering(x.L, succ, (1 << x.L) - 1) == [0, 8]



def brute_cells(x, succ):
    """Every cell of the key table from its definition, by enumeration: for state D,
    at most d units, exactly p stages and the link into D over candidate c, the
    smallest (v, j, m, c') over every chain of up-sets from D to {} with its widths,
    tiers and strategies, v the bottleneck stage cost and (j, m, c') the first move."""
    L, Du, unit = x.L, x.D // x.unit, x.unit
    K = Du.bit_length()
    G = [int(g) for g in x.tierG]
    cand = [int(c) for c in x.cand]
    C = len(cand)
    full = (1 << L) - 1
    st = [int(v) for v in O.lattice_states(x, succ)]
    E = len(st) - 1
    memo = {}

    def tau(D, Dp, m, pos):
        if (D, Dp, m) not in memo:
            memo[(D, Dp, m)] = [O.lattice_terms(x, succ, D, Dp, m, s) for s in range(len(x.strat))]
        ok = [t["tau"] for t in memo[(D, Dp, m)] if t["valid"] and t["tau"] < CAP and t["pmax"] >= pos]
        return min(ok) if ok else None

    def link(D, c):
        if D in (0, full):
            return 0
        byt = sum(int(x.ao[l]) for l in entering(L, succ, D))
        return int(x.tierLat[cand[c]]) + -(-byt * 1000 // int(x.tierBw[cand[c]]))

    def plans(D, p):
        """(units, first stage cost without its incoming link, worst later stage,
        first width m, first move) for every plan of p stages from D."""
        for j, D1 in enumerate(st):
            if D1 == D or (D1 & ~D) or (D1 == 0) != (p == 1):
                continue
            for m in range(K):
                t = tau(D, D1, m, p)
                if t is None:
                    continue
                if D1 == 0:
                    yield 1 << m, t, 0, m, (j, m, 0)
                    continue
                for c2 in range(C):
                    if 2 * (unit << m) > G[cand[c2]]:
                        continue
                    for u, f1, r1, m1, _ in plans(D1, p - 1):
                        if 2 * (unit << m1) > G[cand[c2]]:
                            continue
                        yield (1 << m) + u, t + link(D1, c2), max(f1 + link(D1, c2), r1), m, (j, m, c2)

    want = np.full((len(st), Du + 1, x.Pmax + 1, C), INF, dtype=np.uint64)
    want[E, :, 0, :] = 0
    for i, D in enumerate(st[:-1]):
        for p in range(1, x.Pmax + 1):
            for u, first, rest, m0, (j, m, c2) in plans(D, p):
                for c in range(1 if i == 0 else C):
                    if i > 0 and 2 * (unit << m0) > G[cand[c]]:
                        continue
                    v = max(first + (link(D, c) if i > 0 else 0), rest)
                    if v >= CAP:
                        continue
                    key = (v << 24) | (j << 8) | (m << 4) | c2
                    for d in range(u, Du + 1):
                        if key < int(want[i, d, p, c]):
                            want[i, d, p, c] = key
    return want


def roomy(seed):
    """A tiny DAG with four devices on two tiers (pairs and the whole group), the
    plain strategy always available and, on odd seeds, memory to spare: most cells
    of its table are reachable."""
    x, succ = tiny(seed, Lmax=5)
    x.D, x.unit, x.Pmax = 4, 1, 3
    x.M = max(x.M, x.Pmax)
    x.tierG = np.asarray([2, 8], np.int64)
    x.tierBw = np.asarray([5000 + 997 * (seed % 7), 1500], np.int64)
    x.tierLat = np.asarray([100 * (seed % 5), 2000], np.int64)
    x.cand = np.asarray([0, 1], np.int32)
    x.strat = np.unique(np.vstack([np.asarray([[1, 1, 1, 0, 0]], np.int16), x.strat]), axis=0)
    if seed % 2:
        x.budget = 10**12
    return x, succ


@pytest.mark.parametrize("chunk", range(3))
def test_every_table_cell_matches_enumeration(chunk):
    nonempty = 0
    for seed in range(chunk * 30, (chunk + 1) * 30):
        x, succ = roomy(seed + 12000)
        r = O.solve_lattice(x, succ, want_dp=True)
        want = brute_cells(x, succ)
        assert np.array_equal(r["dp"], want), seed
        nonempty += int(np.count_nonzero(want[:-1] != INF))
    assert nonempty > 1000


@pytest.mark.parametrize("seed", range(20))
def test_pair_tables_cover_every_pair_of_states(seed):
    x, succ = tiny(seed + 1500, Lmax=6)
    st = [int(v) for v in O.lattice_states(x, succ)]
    cost, loads = O.lattice_pair_tables(x, succ)
    K = (x.D // x.unit).bit_length()
    pairs, ld = O.lattice_loads(x, succ)
    want = dict(zip(pairs, ld))
    q = 0
    for i in range(len(st)):
        for j in range(i + 1, len(st)):
            nested = not (st[j] & ~st[i])
            assert nested == ((i, j) in want)
            if nested:
                np.testing.assert_array_equal(loads[q], want[(i, j)])
                for m in range(K):
                    for s in range(len(x.strat)):
                        t = O.lattice_terms(x, succ, st[i], st[j], m, s)
                        w = INF if not t["valid"] or t["tau"] >= CAP else (t["tau"] << 8) | t["pmax"]
                        assert int(cost[q, m, s]) == w
            else:
                assert (cost[q] == INF).all() and (loads[q] == INF).all()
            q += 1
    # a chain's tables are the chain oracle's
    y = synth.random_tiny(seed + 1600, Lmax=7)
    c2, l2 = O.lattice_pair_tables(y, synth.chain_succ(y.L))
    np.testing.assert_array_equal(c2, O.cost_tensor(y))
    np.testing.assert_array_equal(l2, O.loads(y))


def test_widest_graph_chain_of_63_layers():
    # 63 layers is the widest graph (64-bit masks, the top bit stays clear)
    x = synth.config_instance(2, 5)
    x.L = 63
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(x, f, np.resize(getattr(x, f), 63))
    x.Pmax = 8
    st = O.lattice_states(x, synth.chain_succ(63))
    assert len(st) == 64 and int(st[0]) == (1 << 63) - 1
    a, b = O.solve(x, want_dp=True), O.solve_lattice(x, synth.chain_succ(63), want_dp=True)
    assert a["status"] == 0 and a["plan"] == b["plan"] and np.array_equal(a["dp"], b["dp"])
    x.L = 64
    for f in ("fl", "pd", "pe", "ao", "aw", "a2a", "moe"):
        setattr(x, f, np.resize(getattr(x, f), 64))
    assert O.solve_lattice(x, synth.chain_succ(64))["status"] == 2
