"""Pins for the torus tier mapping (Nest Appendix C: hop-distance classes on a mesh
or torus become the tiers of the DP).

The generator's closed form for the diameter of a block of chips on a torus is
checked against brute force over every pair of chips; each tier's group size is
checked to be the largest power-of-two block within its hop limit; and the DP on
small torus clusters is checked against exhaustive enumeration of plans.
"""
import itertools

import numpy as np
import pytest

import brute
from memory_aware_device_gb300 import synth
from oracle import oracle as O

SHAPES = [(2, 2, 2), (4, 4, 1), (4, 2, 2), (4, 4, 4), (8, 2, 1), (8, 8, 1), (2, 1, 1)]


def brute_diameter(shape, block):
    chips = list(itertools.product(*[range(a) for a in block]))
    best = 0
    for p in chips:
        for q in chips:
            d = sum(min(abs(a - b), n - abs(a - b)) for a, b, n in zip(p, q, shape))
            best = max(best, d)
    return best


@pytest.mark.parametrize("shape", SHAPES)
def test_block_diameter_closed_form(shape):
    for block in itertools.product(*[[a for a in (1, 2, 4, 8) if a <= n] for n in shape]):
        assert synth.torus_block_diameter(shape, block) == brute_diameter(shape, block), block


@pytest.mark.parametrize("shape", SHAPES)
def test_tiers_are_the_largest_blocks_per_hop_class(shape):
    G, bw, lat = synth.torus_tiers(shape)
    N = int(np.prod(shape))
    assert list(G) == sorted(set(int(g) for g in G)) and all(g & (g - 1) == 0 for g in G)
    assert G[-1] == N
    for g, h in zip(G[:-1], (1, 2)):
        within = [int(np.prod(b)) for b in itertools.product(*[[a for a in (1, 2, 4, 8) if a <= n] for n in shape])
                  if brute_diameter(shape, b) <= h and int(np.prod(b)) < N]
        assert g == max(within)
    assert bw[-1] < bw[0] and lat[-1] > lat[0]   # the remote class is the slow one


@pytest.mark.parametrize("chunk", range(3))
def test_dp_on_small_tori_matches_exhaustive_enumeration(chunk):
    for seed in range(chunk * 100, (chunk + 1) * 100):
        x = synth.random_tiny(seed + 70000, Lmax=6, Dmax=8)
        shape = ((2, 2, 2), (4, 2, 1), (8, 1, 1))[seed % 3]
        G, bw, lat = synth.torus_tiers(shape)
        if G[-1] < x.D:
            continue
        x.tierG, x.tierBw, x.tierLat = G, bw, lat
        x.cand = np.arange(len(G), dtype=np.int32)
        assert O.validate(x) == 0
        w, X = O.cost_tensor(x), O.links(x)
        b = brute.brute_optimum(x, w, X)
        r = O.solve(x)
        if b is None:
            assert r["status"] == 1
            continue
        assert r["status"] == 0 and (r["t_batch"], len(r["plan"]), r["bottleneck"]) == b


def test_torus_workload_is_valid():
    x = synth.torus_instance(0)
    assert O.validate(x) == 0 and list(x.tierG) == [2, 4, 64] and x.D == 64
