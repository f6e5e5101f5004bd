"""Seeded synthetic placement problems for the Nest placement dynamic program.

Nest: Network- and Memory-Aware Device Placement for Distributed Deep Learning
evaluates on Llama2-7B, Llama3-70B, BertLarge, GPT3-35B/175B and Mixtral-8x7B
(§5.1) over node / rack / spine tiers (§5.2, §5.3, Appendix B).  None of those
models or clusters exist here, so this module draws layer tables, tier tables,
candidate lists and strategy lists shaped like them: transformer blocks with the
usual per-block flop, parameter and activation sizes, tiers of 8-device nodes,
racks and pods, and the strategy grid TP x CP x EP x ZeRO x recompute.

This module holds none of the method's arithmetic: it only draws inputs.  Both the
GPU path and the CPU oracle read the `Instance` objects it returns.

Units: flops per microbatch, bytes, bandwidth in bytes per microsecond, latency
in nanoseconds, device rate R in flop per nanosecond.
"""
from __future__ import annotations

import dataclasses
import itertools
from typing import List, Sequence

import numpy as np

GB = 10**9
SEQ = 2048          # sequence length of one microbatch (microbatch size 1, §5.1)
R_DEFAULT = 10**6   # flop per ns per device
M_DEFAULT = 4096    # microbatches per iteration: global batch 4096 / microbatch 1 (§5.1)
OPT_FACTOR = 6      # optimizer-state bytes per bf16 weight byte (fp32 master + Adam m, v)
AW_FACTOR = 17      # working activation bytes = 17 x the block's output activation bytes


@dataclasses.dataclass
class Instance:
    """One placement problem: a layer chain (or DAG), a tiered cluster and a strategy list."""
    L: int
    D: int
    unit: int
    Pmax: int
    R: int
    M: int
    budget: int
    opt_factor: int
    fl: np.ndarray      # int64 [L] forward flops per microbatch
    pd: np.ndarray      # int64 [L] dense parameter bytes (bf16)
    pe: np.ndarray      # int64 [L] expert parameter bytes, all experts (bf16)
    ao: np.ndarray      # int64 [L] output activation bytes per microbatch
    aw: np.ndarray      # int64 [L] working activation bytes per microbatch
    a2a: np.ndarray     # int64 [L] bytes moved by one all-to-all per microbatch
    moe: np.ndarray     # uint8 [L] 1 for a mixture-of-experts block
    tierG: np.ndarray   # int64 [T] devices per group of tier tau (powers of two)
    tierBw: np.ndarray  # int64 [T] bytes per microsecond
    tierLat: np.ndarray  # int64 [T] nanoseconds
    cand: np.ndarray    # int32 [C] candidate tiers for links between stages
    strat: np.ndarray   # int16 [S, 5] strategies (t, cp, e, z, r)
    schedule: int = 0   # pipeline schedule: 0 = 1F1B, 1 = GPipe
    succ: np.ndarray | None = None   # uint64 [L] successor masks of a layer DAG; None = chain

    @property
    def T(self) -> int:
        return int(self.tierG.shape[0])

    @property
    def C(self) -> int:
        return int(self.cand.shape[0])

    @property
    def S(self) -> int:
        return int(self.strat.shape[0])

    @property
    def Du(self) -> int:
        return self.D // self.unit


def strategy_grid(ts=(1, 2, 4, 8), cps=(1,), es=(1,), zs=(0,), rs=(0,)) -> np.ndarray:
    """All (t, cp, e, z, r) tuples, t outermost and r innermost."""
    rows = list(itertools.product(ts, cps, es, zs, rs))
    return np.asarray(rows, dtype=np.int16).reshape(-1, 5)


def _dense_block(h: int):
    ao = SEQ * h * 2
    return dict(fl=24 * SEQ * h * h, pd=12 * h * h * 2, pe=0, ao=ao,
                aw=AW_FACTOR * ao, a2a=0, moe=0)


def _moe_block(h: int, cf_milli: int, experts: int = 64, topk: int = 2):
    ao = SEQ * h * 2
    # attention 4h^2 parameters dense; each expert is an FFN with 8h^2 parameters
    return dict(fl=(8 + 16 * topk) * SEQ * h * h, pd=4 * h * h * 2,
                pe=experts * 8 * h * h * 2, ao=ao, aw=AW_FACTOR * ao,
                a2a=(SEQ * topk * h * 2 * cf_milli) // 1000, moe=1)


def _layers(blocks) -> dict:
    keys = ("fl", "pd", "pe", "ao", "aw", "a2a")
    out = {k: np.asarray([b[k] for b in blocks], dtype=np.int64) for k in keys}
    out["moe"] = np.asarray([b["moe"] for b in blocks], dtype=np.uint8)
    return out


def _tiers(G, bw_gbs, lat_us, rng=None, sigma=0.0):
    G = np.asarray(G, dtype=np.int64)
    bw = np.asarray([round(b * 1000) for b in bw_gbs], dtype=np.float64)   # GB/s -> B/us
    lat = np.asarray([l * 1000 for l in lat_us], dtype=np.float64)          # us -> ns
    if sigma > 0.0:
        bw = bw * np.exp(rng.normal(0.0, sigma, size=bw.shape))
        lat = lat * np.exp(rng.normal(0.0, sigma, size=lat.shape))
    bw = np.maximum(np.rint(bw), 1000).astype(np.int64)
    lat = np.rint(lat).astype(np.int64)
    return G, bw, lat


def _instance(layers, G, bw, lat, cand, strat, D, unit, Pmax, budget,
              R=R_DEFAULT, M=M_DEFAULT, opt=OPT_FACTOR) -> Instance:
    return Instance(L=int(layers["fl"].shape[0]), D=D, unit=unit, Pmax=Pmax, R=R, M=M,
                    budget=int(budget), opt_factor=opt, tierG=G, tierBw=bw, tierLat=lat,
                    cand=np.asarray(cand, dtype=np.int32), strat=strat, **layers)


# ----------------------------------------------------------------------------------
# The five standard workloads.
# ----------------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny-8L-8dev",
    2: "dense-32L-h4096-64dev",
    3: "dense-96L-h12288-1024dev-oversubscribed",
    4: "moe-48L-h4096-512dev",
    5: "mixed-128L-4096dev-stress",
}
CONFIG_BATCH = {1: 1, 2: 16, 3: 64, 4: 256, 5: 1024}


def config_instance(cfg: int, b: int) -> Instance:
    """Instance b of standard workload cfg (1..5); seed 0 for cfg 1, 1000*cfg+b otherwise."""
    seed = 0 if cfg == 1 else 1000 * cfg + b
    rng = np.random.default_rng(seed)
    if cfg == 1:
        L = 8
        fl = rng.integers(10**9, 10**10 + 1, size=L)
        pd = rng.integers(10**7, 10**8 + 1, size=L)
        ao = rng.integers(10**6, 10**7 + 1, size=L)
        layers = dict(fl=fl.astype(np.int64), pd=pd.astype(np.int64),
                      pe=np.zeros(L, np.int64), ao=ao.astype(np.int64),
                      aw=ao.astype(np.int64).copy(), a2a=np.zeros(L, np.int64),
                      moe=np.zeros(L, np.uint8))
        G, bw, lat = _tiers([8], [900], [2])
        return _instance(layers, G, bw, lat, [0], strategy_grid(zs=(0, 3)),
                         D=8, unit=1, Pmax=8, budget=80 * GB)
    if cfg == 2:
        layers = _layers([_dense_block(4096)] * 32)
        G, bw, lat = _tiers([8, 32, 64], [900, 50, 25], [2, 5, 10])
        budget = 80 * GB if b == 0 else int(rng.integers(40 * GB, 180 * GB + 1))
        return _instance(layers, G, bw, lat, [0, 2], strategy_grid(zs=(0, 1, 3)),
                         D=64, unit=1, Pmax=16, budget=budget)
    if cfg == 3:
        layers = _layers([_dense_block(12288)] * 96)
        G, bw, lat = _tiers([8, 256, 512, 1024], [900, 50, 25, 6.25], [2, 5, 10, 10],
                            rng=rng, sigma=0.2)
        return _instance(layers, G, bw, lat, [0, 1, 2, 3],
                         strategy_grid(cps=(1, 2, 4), zs=(0, 1, 3)),
                         D=1024, unit=8, Pmax=16, budget=80 * GB)
    if cfg == 4:
        cf = int(rng.integers(1000, 2001))
        blocks = [_dense_block(4096) if l % 2 == 0 else _moe_block(4096, cf) for l in range(48)]
        G, bw, lat = _tiers([8, 128, 512], [900, 50, 25], [2, 5, 10])
        strat = strategy_grid(es=(1, 2, 4, 8, 16, 32, 64), zs=(0, 3))
        return _instance(_layers(blocks), G, bw, lat, [0, 1, 2], strat,
                         D=512, unit=8, Pmax=16, budget=80 * GB)
    if cfg == 5:
        h = int(rng.choice([4096, 8192, 16384]))
        cf = int(rng.integers(1000, 2001))
        blocks = [_dense_block(h) if l % 2 == 0 else _moe_block(h, cf) for l in range(128)]
        G, bw, lat = _tiers([8, 128, 1024, 4096], [900, 50, 25, 12.5], [2, 5, 10, 20],
                            rng=rng, sigma=0.2)
        strat = strategy_grid(cps=(1, 2, 4), es=(1, 2, 4, 8, 16, 32, 64),
                              zs=(0, 1, 2, 3), rs=(0, 1))
        budget = int(rng.integers(40 * GB, 180 * GB + 1))
        return _instance(_layers(blocks), G, bw, lat, [0, 1, 2, 3], strat,
                         D=4096, unit=8, Pmax=16, budget=budget)
    raise ValueError(f"unknown workload {cfg}")


def config_batch(cfg: int, B: int | None = None, first: int = 0) -> List[Instance]:
    """Instances first .. first+B-1 of standard workload cfg (B defaults to its batch)."""
    if B is None:
        B = CONFIG_BATCH[cfg] - first
    return [config_instance(cfg, first + b) for b in range(B)]


# ----------------------------------------------------------------------------------
# Tiny random instances: small enough for exhaustive enumeration of every plan.
# ----------------------------------------------------------------------------------

def random_tiny(seed: int, Lmax: int = 6, Dmax: int = 8, Tmax: int = 3, Cmax: int = 3,
                Smax: int = 8) -> Instance:
    """A small random problem with tight memory and uneven links.

    Values are small integers so that ties, rounding and infeasibility all occur.
    """
    rng = np.random.default_rng(10**6 + seed)
    L = int(rng.integers(1, Lmax + 1))
    unit = int(rng.choice([1, 1, 2]))
    Du = int(rng.integers(1, Dmax // unit + 1))
    D = Du * unit
    T = int(rng.integers(1, Tmax + 1))
    # strictly increasing powers of two, the top one at least D
    top = max(1, int(2 ** np.ceil(np.log2(max(D, 1)))))
    exps = sorted(rng.choice(np.arange(0, int(np.log2(top)) + 1), size=min(T, int(np.log2(top)) + 1),
                             replace=False).tolist())
    exps[-1] = int(np.log2(top)) + int(rng.integers(0, 2))
    exps = sorted(set(exps))
    G = np.asarray([2 ** x for x in exps], dtype=np.int64)
    T = G.shape[0]
    bw = rng.integers(1000, 20000, size=T).astype(np.int64)
    lat = rng.integers(0, 3000, size=T).astype(np.int64)
    C = int(rng.integers(1, min(Cmax, T) + 1))
    cand = np.sort(rng.choice(np.arange(T), size=C, replace=False)).astype(np.int32)
    moe = (rng.random(L) < 0.4).astype(np.uint8)
    fl = rng.integers(0, 4 * 10**6, size=L).astype(np.int64)
    pd = rng.integers(0, 3 * 10**5, size=L).astype(np.int64)
    pe = (rng.integers(0, 6 * 10**5, size=L) * moe).astype(np.int64)
    ao = rng.integers(0, 2 * 10**5, size=L).astype(np.int64)
    aw = (ao * rng.integers(1, 6, size=L)).astype(np.int64)
    a2a = (rng.integers(0, 2 * 10**5, size=L) * moe).astype(np.int64)
    pool = list(itertools.product((1, 2, 4), (1, 2), (1, 2, 4), (0, 1, 2, 3), (0, 1)))
    S = int(rng.integers(1, Smax + 1))
    idx = rng.choice(len(pool), size=S, replace=False)
    strat = np.asarray([pool[i] for i in idx], dtype=np.int16).reshape(-1, 5)
    Pmax = int(rng.integers(1, 7))
    M = int(rng.integers(Pmax, Pmax + 40))
    R = int(rng.integers(1, 50))
    budget = int(rng.integers(0, 6 * 10**6))
    return Instance(L=L, D=D, unit=unit, Pmax=Pmax, R=R, M=M, budget=budget,
                    opt_factor=int(rng.integers(0, 7)), fl=fl, pd=pd, pe=pe, ao=ao, aw=aw,
                    a2a=a2a, moe=moe, tierG=G, tierBw=bw, tierLat=lat, cand=cand, strat=strat)


# Joint microbatch-size exploration (Nest §5.2.3: the microbatch size is explored
# together with the placement).  The workloads above use microbatches of one
# sample; a variant with b samples per microbatch scales every per-microbatch
# quantity (flops, activations, all-to-all volume) by b and runs M = global batch / b
# microbatches per iteration; parameters do not change.
MICROBATCH_SIZES = (1, 2, 4, 8)
GLOBAL_BATCH = 4096


def microbatch_variant(inst: Instance, mbs: int, global_batch: int = GLOBAL_BATCH) -> Instance:
    """The instance with `mbs` samples per microbatch (inst has one)."""
    y = dataclasses.replace(inst)
    y.fl, y.ao, y.aw, y.a2a = (np.asarray(a, np.int64) * mbs for a in (inst.fl, inst.ao, inst.aw, inst.a2a))
    y.M = max(global_batch // mbs, inst.Pmax)
    return y


def joint_batch(problems: Sequence[Instance], sizes=MICROBATCH_SIZES) -> List[Instance]:
    """Every problem expanded into its microbatch variants, consecutively."""
    return [microbatch_variant(x, b) for x in problems for b in sizes]


# Torus and mesh clusters (Nest Appendix C, §4 "non-uniform mesh"): tiers are
# hop-distance classes - direct neighbours, two hops, and the rest ("remote", behind
# slower inter-mesh links).  For the DP a tier is a group size G (a power of two),
# a bandwidth and a latency: G_t is the largest power-of-two block of chips whose
# torus diameter is within the class's hop distance, the latency is that many hops,
# and the remote class reaches every chip.

def torus_block_diameter(shape, block) -> int:
    """Largest hop distance between two chips of an axis-aligned block on a torus
    (wrap-around links on every axis): along an axis of length n, a block of a chips
    spans a - 1 hops, or floor(n / 2) when it covers the whole ring."""
    d = 0
    for n, a in zip(shape, block):
        d += n // 2 if a == n else a - 1
    return d


def _blocks(shape, g):
    """Axis-aligned blocks of g chips that fit in the torus (power-of-two sides)."""
    sides = [[a for a in (1 << k for k in range(12)) if a <= n] for n in shape]
    for block in itertools.product(*sides):
        if int(np.prod(block)) == g:
            yield block


def torus_tiers(shape=(4, 4, 4), hops=(1, 2), link_gbs=50.0, hop_us=1.0, remote_gbs=12.5, remote_us=5.0):
    """(G, bandwidth, latency) arrays for the hop classes of a torus: for each hop
    limit h the largest power-of-two block of diameter <= h, then the whole torus."""
    N = int(np.prod(shape))
    best = {}   # g -> smallest diameter of a g-chip block
    g = 1
    while g <= N:
        ds = [torus_block_diameter(shape, b) for b in _blocks(shape, g)]
        if ds:
            best[g] = min(ds)
        g *= 2
    G, bw, lat = [], [], []
    for h in hops:
        fit = [g for g, d in best.items() if d <= h and g < N]
        if fit and (not G or max(fit) > G[-1]):
            G.append(max(fit))
            bw.append(link_gbs)
            lat.append(h * hop_us)
    G.append(N)
    bw.append(remote_gbs)
    lat.append(remote_us)
    return _tiers(G, bw, lat)


TORUS_NAME = "dense-32L-h4096-64chip-torus4x4x4"


def torus_instance(b: int, shape=(4, 4, 4)) -> Instance:
    """Workload 2's model and budgets on a 4x4x4 torus of 64 chips: tiers are the
    1-hop pairs, the 2-hop 2x2 squares and the whole torus (remote)."""
    x = config_instance(2, b)
    G, bw, lat = torus_tiers(shape)
    x.tierG, x.tierBw, x.tierLat = G, bw, lat
    x.cand = np.arange(len(G), dtype=np.int32)
    return x


# ----------------------------------------------------------------------------------
# Layer DAGs (Nest §4 states Eq. 3 over downsets of the operator graph).  A graph is
# given by successor masks: bit v of succ[l] is set for each edge l -> v, and the
# layers are numbered topologically (v > l).
# ----------------------------------------------------------------------------------

def chain_succ(L: int) -> np.ndarray:
    """The successor masks of the chain 0 -> 1 -> ... -> L-1."""
    return np.asarray([(1 << (l + 1)) if l + 1 < L else 0 for l in range(L)], dtype=np.uint64)


def random_dag(seed: int, L: int, density: float) -> np.ndarray:
    """Each forward edge u -> v (u < v) present with probability `density`."""
    rng = np.random.default_rng(2 * 10**6 + seed)
    succ = np.zeros(L, dtype=np.uint64)
    for u in range(L):
        for v in range(u + 1, L):
            if rng.random() < density:
                succ[u] |= np.uint64(1 << v)
    return succ


def two_tower_succ(branch: int = 8, trunk: int = 16) -> np.ndarray:
    """Two encoder branches of `branch` blocks each feeding a shared trunk of `trunk`
    blocks: branch A is layers [0, branch), branch B [branch, 2 branch), the trunk
    the rest; both branch ends feed the first trunk block."""
    L = 2 * branch + trunk
    succ = np.zeros(L, dtype=np.uint64)
    for base in (0, branch):
        for l in range(base, base + branch - 1):
            succ[l] = np.uint64(1 << (l + 1))
        succ[base + branch - 1] = np.uint64(1 << (2 * branch))
    for l in range(2 * branch, L - 1):
        succ[l] = np.uint64(1 << (l + 1))
    return succ


TWO_TOWER_NAME = "two-tower-32L-h4096-64dev"


def two_tower_instance(b: int) -> Instance:
    """Workload 2's blocks, tiers and budgets arranged as two 8-block encoder branches
    feeding a 16-block trunk (97 up-sets)."""
    x = config_instance(2, b)
    x.succ = two_tower_succ()
    return x
