"""Helpers for GPU parity tests: run the CUDA path and read its intermediate tables."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from memory_aware_device_gb300 import build as nbuild
from memory_aware_device_gb300 import nest
from oracle import oracle as O

U64 = np.uint64


def ensure_built():
    nbuild.build()
    O.build()


def run(instances, chunk=0, cluster=0, jsplit=0, spin_limit=0, Pcap=None, Dumax=None, variant=0,
        keep_costs=True, Vmax=None):
    """Solve on cuda:0 (keeping the stage-cost tensor for inspection unless told
    otherwise); returns (solver, results)."""
    import torch
    dims = nest.make_dims(instances, Pcap=Pcap, Dumax=Dumax, Vmax=Vmax)
    s = nest.Solver(dims, chunk=chunk, keep_costs=keep_costs)
    s.load(nest.pack_records(instances, dims))
    s.run(opt=nest.options(chunk=chunk, cluster=cluster, jsplit=jsplit, spin_limit=spin_limit,
                           variant=variant, keep_costs=keep_costs))
    torch.cuda.synchronize()
    return s, s.results()


def last_state(inst):
    """Index of the empty state: L for a chain, the up-set count less one for a graph."""
    succ = getattr(inst, "succ", None)
    return int(inst.L) if succ is None else nest.upset_count(succ) - 1


def _slice(ws, off, count, dtype):
    b = np.dtype(dtype).itemsize
    return ws[off:off + count * b].cpu().numpy().view(dtype)


def cost_table(s, b, inst):
    lay = nest.workspace_layout(s.dims, s.chunk)
    per = lay.NP * lay.Kmax * lay.Spad
    t = _slice(s.workspace, lay.cost + 8 * per * b, per, U64).reshape(lay.NP, lay.Kmax, lay.Spad)
    K = (inst.D // inst.unit).bit_length()
    E = last_state(inst)
    return t[:E * (E + 1) // 2, :K, :len(inst.strat)]


def loads_table(s, b, inst):
    lay = nest.workspace_layout(s.dims, s.chunk)
    per = s.dims.Pcap * lay.NP * lay.Kpad
    t = _slice(s.workspace, lay.loads + 8 * per * b, per, U64).reshape(s.dims.Pcap, lay.NP, lay.Kpad)
    K = (inst.D // inst.unit).bit_length()
    E = last_state(inst)
    return np.transpose(t[:inst.Pmax, :E * (E + 1) // 2, :K], (1, 2, 0))   # [pair][m][p-1] like the oracle


def dp_keys(s, b, inst):
    """GPU DP table as packed keys in the oracle's [i][d][p][c] order (p >= 1, i < L)."""
    lay = nest.workspace_layout(s.dims, s.chunk)
    shape = (s.dims.Pcap, lay.N, s.dims.Cmax, lay.Dpad)
    per = int(np.prod(shape))
    v = _slice(s.workspace, lay.dpv + 8 * per * b, per, np.int64).reshape(shape)
    a = _slice(s.workspace, lay.dpa + 4 * per * b, per, np.uint32).reshape(shape)
    Du, C, E = inst.D // inst.unit, len(inst.cand), last_state(inst)
    v = v[:inst.Pmax, :E, :C, :Du + 1].astype(U64)
    a = a[:inst.Pmax, :E, :C, :Du + 1].astype(U64)
    keys = (v << U64(24)) | a
    return np.transpose(keys, (1, 3, 0, 2))   # [i][d][p-1][c]


def oracle_dp_keys(inst, dp):
    return dp[:last_state(inst), :, 1:, :]


def oracle_many(instances, fn=O.solve, threads=None):
    threads = threads or os.cpu_count() or 1
    O.lib()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, instances))


def word_tag_bits(instances):
    """Tag bits of the resident sweep's 32-bit words for a batch: log2 of the widths its
    kernels are instantiated for (4, 8 or 16) when the batch has at most two link
    candidates (packed words), else 0 (plain words)."""
    dims = nest.make_dims(instances)
    kmax = int(dims.Dumax).bit_length()
    kt = 4 if kmax <= 4 else 8 if kmax <= 8 else 16
    return {4: 2, 8: 3, 16: 4}[kt] if dims.Cmax <= 2 else 0


def value_bound(inst):
    """The largest finite per-position load plus twice the largest link cost (each
    saturated at 2^31 - 1), a bound of every finite value of the instance's DP."""
    lo = O.loads(inst)
    fin = lo[lo != np.uint64(2**64 - 1)]
    ml = int((fin >> U64(16)).max()) if fin.size else 0
    mx = int(np.max(O.links(inst)))
    return min(ml, 2**31 - 1) + 2 * min(mx, 2**31 - 1)


def packed_words(inst, tb):
    """Whether the 32-bit words are packed with tb tag bits (tb > 0): the value bound
    is below 2^(32 - tb) - 1."""
    return tb > 0 and value_bound(inst) < 2**(32 - tb) - 1


def narrow_words(inst, tb=0):
    """Whether the resident sweep takes its 32-bit value words for this instance (tb:
    the batch's tag bits): a chain below 2^30 (packed or plain), a graph only when its
    words can be packed (or, with no tag bits, below 2^30)."""
    if getattr(inst, "succ", None) is not None and tb:
        return packed_words(inst, tb)
    return value_bound(inst) < 2**30


def scaled(inst, factor):
    """The same instance with every layer's flops multiplied by `factor`."""
    import copy
    y = copy.deepcopy(inst)
    y.fl = y.fl * factor
    return y


def same_result(g, o):
    return (g["status"] == o["status"] and g["t_batch"] == o["t_batch"] and
            (g["status"] != 0 or (g["bottleneck"] == o["bottleneck"] and g["plan"] == o["plan"])))


def solve_graph(inst):
    return O.solve_lattice(inst, inst.succ)


def check_graph_tables(s, b, inst):
    """Every table of graph instance b against the oracle over up-sets; returns the
    oracle's result."""
    cost, loads = O.lattice_pair_tables(inst, inst.succ)
    np.testing.assert_array_equal(cost_table(s, b, inst), cost)
    np.testing.assert_array_equal(loads_table(s, b, inst), loads)
    o = O.solve_lattice(inst, inst.succ, want_dp=True)
    np.testing.assert_array_equal(dp_keys(s, b, inst), oracle_dp_keys(inst, o["dp"]))
    return o


def same_graph_result(g, o):
    """Results equal, and each stage's layer mask is states[i] minus states[j]."""
    if not same_result(g, o):
        return False
    st = o["states"]
    return g["status"] != 0 or g["layers"] == [int(st[i]) & ~int(st[j]) for i, j, *_ in o["plan"]]


def layered_words(inst):
    """The layered sweep's 32-bit words for an instance, as (mode, tag bits, vmax): rank
    tags (mode 0, log2 of the (m, c') pairs its first stage admits) when the value bound
    is at most their largest exact value, else width tags (mode 1, log2 of the widths)."""
    Du = inst.D // inst.unit
    K = Du.bit_length()
    E = 0
    for c in inst.cand:
        G = int(inst.tierG[int(c)])
        ml = max((m for m in range(16) if 2 * (int(inst.unit) << m) <= G), default=-1)
        if ml >= 0:
            E += min(ml, K - 1) + 1
    tr = 1
    while (1 << tr) < E:
        tr += 1
    tw = 1
    while (1 << tw) < K:
        tw += 1
    vb = value_bound(inst)
    mode = 0 if vb <= 2**(32 - tr) - 3 else 1
    tb = tr if mode == 0 else tw
    return mode, tb, 2**(32 - tb) - 3


def layered_fits(inst):
    """Whether no word of the layered sweep can saturate for the instance (at most four
    candidates and a value bound within its mode's exact values)."""
    _, _, vmax = layered_words(inst)
    return len(inst.cand) <= 4 and value_bound(inst) <= vmax
