"""Python access to the CPU oracle (nest_oracle.c).  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
module.  It marshals `synth.Instance`-like objects (any object with the same
attributes) into the oracle's own C structs; it shares no code with the CUDA
library or its Python binding.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nest_oracle.c")
LIB = os.path.join(HERE, "libnest_oracle.so")
CAP = (1 << 40) - 1
INF = (1 << 64) - 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no machine-specific flags)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


class _Inst(C.Structure):
    _fields_ = [("L", C.c_int32), ("D", C.c_int32), ("unit", C.c_int32), ("T", C.c_int32),
                ("C", C.c_int32), ("S", C.c_int32), ("Pmax", C.c_int32), ("schedule", C.c_int32),
                ("R", C.c_int64), ("M", C.c_int64), ("budget", C.c_int64), ("opt_factor", C.c_int64),
                ("fl", C.c_void_p), ("pd", C.c_void_p), ("pe", C.c_void_p), ("ao", C.c_void_p),
                ("aw", C.c_void_p), ("a2a", C.c_void_p), ("moe", C.c_void_p),
                ("G", C.c_void_p), ("bw", C.c_void_p), ("lat", C.c_void_p),
                ("cand", C.c_void_p), ("strat", C.c_void_p)]


class _Stage(C.Structure):
    _fields_ = [("i", C.c_int32), ("j", C.c_int32), ("k", C.c_int32), ("s", C.c_int32),
                ("c_next", C.c_int32)]


TERM_NAMES = ("valid", "comp", "tp", "cpc", "ep", "z3", "sd", "se", "tau",
              "w", "g", "o", "act", "stash", "stat", "pmax")


class _Terms(C.Structure):
    _fields_ = [(n, C.c_int64) for n in TERM_NAMES]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(LIB)
            P = C.POINTER
            L.or_validate.argtypes = [P(_Inst)]
            L.or_stage_terms.argtypes = [P(_Inst), C.c_int, C.c_int, C.c_int, C.c_int, P(_Terms)]
            L.or_cost_tensor.argtypes = [P(_Inst), C.c_void_p]
            L.or_links.argtypes = [P(_Inst), C.c_void_p]
            L.or_loads.argtypes = [P(_Inst), C.c_void_p]
            L.or_dp_table_words.argtypes = [P(_Inst)]
            L.or_dp_table_words.restype = C.c_int64
            L.or_solve.argtypes = [P(_Inst), C.c_void_p, P(C.c_int64), P(C.c_int64),
                                   P(C.c_int32), P(_Stage)]
            L.or_lattice_states.argtypes = [P(_Inst), C.c_void_p, C.c_void_p]
            L.or_lattice_loads.argtypes = [P(_Inst), C.c_void_p, C.c_void_p, C.c_int, C.c_void_p]
            L.or_lattice_loads.restype = C.c_int64
            L.or_lattice_terms.argtypes = [P(_Inst), C.c_void_p, C.c_uint64, C.c_uint64, C.c_int, C.c_int,
                                           P(_Terms)]
            L.or_lattice_link.argtypes = [P(_Inst), C.c_void_p, C.c_uint64, C.c_int]
            L.or_lattice_link.restype = C.c_int64
            L.or_lattice_cost_tensor.argtypes = [P(_Inst), C.c_void_p, C.c_void_p, C.c_int, C.c_void_p]
            L.or_solve_lattice.argtypes = [P(_Inst), C.c_void_p, C.c_void_p, P(C.c_int64), P(C.c_int64),
                                           P(C.c_int32), P(_Stage)]
            _lib = L
    return _lib


class Marshalled:
    """Keeps the numpy arrays alive while the C struct points into them."""

    def __init__(self, inst):
        def arr(a, dt):
            return np.ascontiguousarray(np.asarray(a, dtype=dt))
        self.keep = {
            "fl": arr(inst.fl, np.int64), "pd": arr(inst.pd, np.int64), "pe": arr(inst.pe, np.int64),
            "ao": arr(inst.ao, np.int64), "aw": arr(inst.aw, np.int64), "a2a": arr(inst.a2a, np.int64),
            "moe": arr(inst.moe, np.uint8), "G": arr(inst.tierG, np.int64),
            "bw": arr(inst.tierBw, np.int64), "lat": arr(inst.tierLat, np.int64),
            "cand": arr(inst.cand, np.int32), "strat": arr(inst.strat, np.int16).reshape(-1, 5),
        }
        k = self.keep
        self.s = _Inst(L=int(inst.L), D=int(inst.D), unit=int(inst.unit), T=len(k["G"]),
                       C=len(k["cand"]), S=k["strat"].shape[0], Pmax=int(inst.Pmax),
                       schedule=int(getattr(inst, "schedule", 0)),
                       R=int(inst.R), M=int(inst.M), budget=int(inst.budget),
                       opt_factor=int(inst.opt_factor),
                       **{n: v.ctypes.data for n, v in k.items()})
        self.K = 0
        while (1 << self.K) <= inst.D // inst.unit:
            self.K += 1
        self.NP = inst.L * (inst.L + 1) // 2


def validate(inst) -> int:
    m = Marshalled(inst)
    return lib().or_validate(C.byref(m.s))


def terms(inst, i: int, j: int, m: int, s: int) -> dict:
    mm = Marshalled(inst)
    t = _Terms()
    lib().or_stage_terms(C.byref(mm.s), i, j, m, s, C.byref(t))
    return {n: int(getattr(t, n)) for n in TERM_NAMES}


def cost_tensor(inst) -> np.ndarray:
    """uint64 [NP, K, S] packed (tau << 8) | pmax, all ones where not applicable."""
    m = Marshalled(inst)
    out = np.empty((m.NP, m.K, m.s.S), dtype=np.uint64)
    lib().or_cost_tensor(C.byref(m.s), out.ctypes.data)
    return out


def links(inst) -> np.ndarray:
    m = Marshalled(inst)
    out = np.empty((inst.L + 1, m.s.C), dtype=np.int64)
    lib().or_links(C.byref(m.s), out.ctypes.data)
    return out


def loads(inst) -> np.ndarray:
    """uint64 [NP, K, Pmax] packed (tau* << 16) | s*, all ones where nothing fits."""
    m = Marshalled(inst)
    out = np.empty((m.NP, m.K, inst.Pmax), dtype=np.uint64)
    lib().or_loads(C.byref(m.s), out.ctypes.data)
    return out


def solve(inst, want_dp: bool = False) -> dict:
    """Optimal batch time, bottleneck stage time and the canonical plan."""
    m = Marshalled(inst)
    dp = None
    dp_ptr = None
    if want_dp:
        Du = inst.D // inst.unit
        dp = np.empty((inst.L + 1, Du + 1, inst.Pmax + 1, m.s.C), dtype=np.uint64)
        dp_ptr = dp.ctypes.data
    t = C.c_int64()
    v = C.c_int64()
    n = C.c_int32()
    stages = (_Stage * 32)()
    st = lib().or_solve(C.byref(m.s), dp_ptr, C.byref(t), C.byref(v), C.byref(n), stages)
    plan = [(stages[q].i, stages[q].j, stages[q].k, stages[q].s, stages[q].c_next)
            for q in range(n.value)]
    return {"status": st, "t_batch": t.value, "bottleneck": v.value, "plan": plan, "dp": dp}


def solve_many(instances, threads: int | None = None) -> list:
    """Solve independent instances on a thread pool (ctypes releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    lib()
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(solve, instances))


def solve_joint(variants) -> dict:
    """Joint search over the variants of one problem (Nest §5.2.3, the microbatch size
    explored together with the placement): the variant with the smallest t_batch, ties
    to the earlier variant; best = -1 when no variant is solved."""
    best, res = -1, None
    results = [solve(v) for v in variants]
    for q, r in enumerate(results):
        if r["status"] == 0 and (best < 0 or r["t_batch"] < res["t_batch"]):
            best, res = q, r
    return {"best": best, "t_batch": res["t_batch"] if res else -1, "results": results}


# ---------------------------------------------------------------------------------
# Layer DAGs: succ[l] is the bit mask of the successors of layer l (layers numbered
# topologically); the states of Eq. 3 are the up-sets of the graph.


def _succ(succ) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(succ, dtype=np.uint64))


def lattice_states(inst, succ) -> np.ndarray | None:
    """The up-sets as layer masks in DP order, or None beyond the lattice limits."""
    m, sc = Marshalled(inst), _succ(succ)
    out = np.zeros(256, dtype=np.uint64)
    n = lib().or_lattice_states(C.byref(m.s), sc.ctypes.data, out.ctypes.data)
    return None if n < 0 else out[:n].copy()


def lattice_loads(inst, succ) -> tuple[list, np.ndarray]:
    """Transitions [(i, j)] in the oracle's order and their loads [T, K, Pmax]."""
    m, sc = Marshalled(inst), _succ(succ)
    st = lattice_states(inst, succ)
    n = lib().or_lattice_loads(C.byref(m.s), sc.ctypes.data, st.ctypes.data, len(st), None)
    out = np.empty((n, m.K, inst.Pmax), dtype=np.uint64)
    lib().or_lattice_loads(C.byref(m.s), sc.ctypes.data, st.ctypes.data, len(st), out.ctypes.data)
    pairs = [(i, j) for i in range(len(st)) for j in range(i + 1, len(st))
             if not (int(st[j]) & ~int(st[i])) and st[j] != st[i]]
    return pairs, out


def lattice_terms(inst, succ, D: int, Dp: int, m: int, s: int) -> dict:
    mm, sc = Marshalled(inst), _succ(succ)
    t = _Terms()
    lib().or_lattice_terms(C.byref(mm.s), sc.ctypes.data, D, Dp, m, s, C.byref(t))
    return {n: int(getattr(t, n)) for n in TERM_NAMES}


def lattice_link(inst, succ, D: int, c: int) -> int:
    mm, sc = Marshalled(inst), _succ(succ)
    return int(lib().or_lattice_link(C.byref(mm.s), sc.ctypes.data, D, c))


def solve_lattice(inst, succ, want_dp: bool = False) -> dict:
    """Eq. 3 over the up-sets of a layer DAG; plan stage i/j are state indices into
    `states`."""
    m, sc = Marshalled(inst), _succ(succ)
    st = lattice_states(inst, succ)
    dp = None
    dp_ptr = None
    if want_dp and st is not None:
        Du = inst.D // inst.unit
        dp = np.empty((len(st), Du + 1, inst.Pmax + 1, m.s.C), dtype=np.uint64)
        dp_ptr = dp.ctypes.data
    t, v, n = C.c_int64(), C.c_int64(), C.c_int32()
    stages = (_Stage * 64)()
    rc = lib().or_solve_lattice(C.byref(m.s), sc.ctypes.data, dp_ptr, C.byref(t), C.byref(v), C.byref(n), stages)
    plan = [(stages[q].i, stages[q].j, stages[q].k, stages[q].s, stages[q].c_next)
            for q in range(n.value)]
    return {"status": rc, "t_batch": t.value, "bottleneck": v.value, "plan": plan, "dp": dp,
            "states": st}


def lattice_pair_tables(inst, succ) -> tuple[np.ndarray, np.ndarray]:
    """Over every pair of states (i, j), i < j, in pair order: the stage-cost words
    [NP, K, S] and the per-position loads [NP, K, Pmax], all ones where state j is
    not inside state i."""
    m, sc = Marshalled(inst), _succ(succ)
    st = lattice_states(inst, succ)
    ns = len(st)
    npairs = ns * (ns - 1) // 2
    cost = np.empty((npairs, m.K, m.s.S), dtype=np.uint64)
    lib().or_lattice_cost_tensor(C.byref(m.s), sc.ctypes.data, st.ctypes.data, ns, cost.ctypes.data)
    pairs, ld = lattice_loads(inst, succ)
    loads = np.full((npairs, m.K, inst.Pmax), INF, dtype=np.uint64)
    for t, (i, j) in enumerate(pairs):
        loads[i * (ns - 1) - i * (i - 1) // 2 + (j - i - 1)] = ld[t]
    return cost, loads
