"""Benchmark of the Nest placement DP on GB300: DP relaxations/s and solves/s.

One step = one nest_solve of a whole batch: prep, stage loads (cost build and
strategy reduction), DP sweep and backtrack, inputs resident in HBM.  The default
workload is the large sweep stress batch: 1024 instances of 128 mixed dense / MoE
layers (hidden 4096, 8192 or 16384) on 4096 devices in four tiers, 672 strategies.
`value` counts the min-max transitions (j, m, c') of the recurrence whose successor
cell can hold a value, per second; `solves_per_s` counts instances.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 5] [--impl ours|reference]

Under torchrun (N > 1) every rank solves its own batch (different seeds): the
work is partitioned, so there is no collective on the data path (weak scaling);
only the timing barrier and the max-over-ranks use the process group.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from memory_aware_device_gb300 import synth  # noqa: E402

METRIC = "DP relaxations/sec and placement solves/sec on 1 GB300; % of HBM roofline"
UNIT = "relaxations/s"
KERNELS = ("prep", "stage_loads", "dp_sweep", "backtrack")
NEV = len(KERNELS) + 1   # events per chunk
KERNEL_SRC = {"prep": ("nest_prep.cu",), "stage_loads": ("nest_loads.cu",),
              "dp_sweep": ("nest_sweep.cu", "nest_sweep_res_a.cu", "nest_sweep_res_b.cu", "nest_layered.cu"),
              "backtrack": ("nest_backtrack.cu",)}
L2_FLUSH_BYTES = 256 << 20


def states(x) -> list:
    """The DP states of an instance as layer masks, in DP order: the suffixes of a
    chain, or the up-sets of a layer DAG by size descending then mask ascending."""
    if getattr(x, "succ", None) is None:
        return [((1 << x.L) - 1) ^ ((1 << i) - 1) for i in range(x.L + 1)]
    succ = [int(v) for v in x.succ]
    out, stack = [], [(x.L - 1, 0)]
    while stack:
        l, D = stack.pop()
        if l < 0:
            out.append(D)
            continue
        stack.append((l - 1, D))
        if succ[l] & ~D == 0:
            stack.append((l - 1, D | (1 << l)))
    return sorted(out, key=lambda D: (-bin(D).count("1"), D))


def _pairs(x):
    """(E, per-state layer counts, nested[i] = bool array over states j, moe_in[i] =
    bool array: the stage from state i to state j holds a MoE layer)."""
    if getattr(x, "succ", None) is None:
        L = x.L
        pm = np.concatenate([[0], np.cumsum(np.asarray(x.moe, dtype=np.int64))])
        sizes = [L - i for i in range(L + 1)]
        nested = [np.arange(L + 1) > i for i in range(L + 1)]
        moe_in = [(pm - pm[i]) > 0 for i in range(L + 1)]
        return L, sizes, nested, moe_in
    st = np.asarray(states(x), dtype=np.uint64)
    mm = np.uint64(sum(1 << l for l in range(x.L) if int(x.moe[l])))
    sizes = [bin(int(v)).count("1") for v in st]
    idx = np.arange(len(st))
    nested = [(idx > i) & ((st & ~st[i]) == 0) for i in range(len(st))]
    moe_in = [((st[i] & ~st) & mm) != 0 for i in range(len(st))]
    return len(st) - 1, sizes, nested, moe_in


def _count(x, with_strategies: bool) -> int:
    Du, P, C, u = x.D // x.unit, x.Pmax, len(x.cand), x.unit
    G = [int(x.tierG[c]) for c in x.cand]
    K = Du.bit_length()
    E, sizes, nested, moe_in = _pairs(x)
    sizes = np.asarray(sizes)
    # strategies valid for a stage of width unit * 2^m, without / with a MoE layer
    nvalid = np.ones((K, 2), dtype=np.int64)
    if with_strategies:
        for m in range(K):
            k = u << m
            for hm in (0, 1):
                nvalid[m, hm] = sum(1 for t, cp, e, _, _ in x.strat
                                    if not (k % (int(t) * int(cp)) or (k // (int(t) * int(cp))) % int(e)
                                            or (int(e) > 1 and not hm)))
    tot = 0
    for i in range(E):
        Pi = min(P, sizes[i])
        inner_j = nested[i].copy()
        inner_j[E] = False
        for m in range(K):
            k = u << m
            w = nvalid[m][moe_in[i].astype(np.int64)]
            last = int(w[E])
            ncp = sum(1 for g in G if 2 * k <= g)
            # position p >= 2 relaxes cut point j only when state j can still hold the
            # p - 1 stages after it, and width 2^m only when d - 2^m >= p - 1 units remain
            # for them: otherwise the successor cell dp[j][d - 2^m][p - 1] has no value
            n_after = 0
            for p in range(2, Pi + 1):
                nd = Du - (1 << m) - (p - 1) + 1
                if nd <= 0:
                    break
                n_after += nd * int(w[inner_j & (sizes >= p - 1)].sum())
            for c in range(1 if i == 0 else C):
                if i > 0 and 2 * k > G[c]:
                    continue
                tot += (Du - (1 << m) + 1) * last + n_after * ncp
    return tot


_COUNTS = {}


def _structure(x, with_strategies: bool):
    """What the work counts depend on: instances of one workload share it."""
    key = (int(x.L), int(x.D), int(x.unit), int(x.Pmax), tuple(int(x.tierG[int(c)]) for c in x.cand),
           None if getattr(x, "succ", None) is None else tuple(int(v) for v in x.succ))
    if with_strategies:
        key += (tuple(map(tuple, np.asarray(x.strat).tolist())), tuple(int(v) for v in x.moe))
    return key


def _count_cached(x, with_strategies: bool) -> int:
    key = (with_strategies,) + _structure(x, with_strategies)
    if key not in _COUNTS:
        _COUNTS[key] = _count(x, with_strategies)
    return _COUNTS[key]


def relaxations(x) -> int:
    """Min-max transitions (j, m, c') of the recurrence for one instance whose
    successor cell can hold a value: every cell (i, d, p, c) times its cut points j
    (states inside state i with at least p - 1 layers), widths 2^m <= d - (p - 1)
    allowed by the link tier, and next-link candidates c' allowed for that width.
    Transitions into successor cells that are empty by construction (too few layers
    or device units left for the remaining p - 1 stages) are not counted."""
    return _count_cached(x, False)


def relaxations_with_strategies(x) -> int:
    """The same transitions counted with the strategy axis, (j, m, s, c'): every
    relaxation times the strategies valid for its stage and width (t cp divides the
    width, e divides the data-parallel degree, e > 1 only over a MoE layer) - the
    work of the recurrence before the strategy minimum is hoisted out of it."""
    return _count(x, True)


def state_pairs(x) -> int:
    E = len(states(x)) - 1
    return E * (E + 1) // 2


def cost_words(x) -> int:
    return state_pairs(x) * (x.D // x.unit).bit_length() * len(x.strat)


def oracle_solve(x):
    from oracle import oracle as O
    return O.solve(x) if getattr(x, "succ", None) is None else O.solve_lattice(x, x.succ)


def src_hash(kernel: str) -> str:
    """Hash of a kernel's source files and every header the kernels share."""
    d = os.path.join(ROOT, "memory_aware_device_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SRC[kernel]:
        h.update(open(os.path.join(d, f), "rb").read())
    for f in sorted(os.listdir(d)):
        if f.endswith(".cuh"):
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


# Plain integer ALU peak for the sweep's relaxation: 152 SMs x 128 INT32 lanes per
# clock, and 11 INT32 instructions for the minimal op mix of one relaxation
# (64-bit add: 2, 64-bit max: 4, 64-bit compare: 2, select of value and argument: 3).
SMS, INT32_LANES, OPS_PER_RELAX = 152, 128, 11


def alu_peak_relax_per_s(sm_mhz):
    return SMS * INT32_LANES * sm_mhz * 1e6 / OPS_PER_RELAX


def measured_relax_peak(wide: int = 0):
    """Relaxations/s of the relaxation arithmetic alone (one max, one compare, two
    selects per candidate and cell, values in registers, every SM busy), from the
    microbenchmark built next to the library; None if it cannot run."""
    try:
        from memory_aware_device_gb300 import build as nbuild
        lib = ctypes.CDLL(nbuild.build_peak())
        lib.nest_peak_relax.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        out = ctypes.c_double()
        return out.value if lib.nest_peak_relax(wide, 4096, ctypes.byref(out)) == 0 else None
    except (OSError, RuntimeError):
        return None


def relax_peak_mode(instances, plan) -> int:
    """Which relaxation peak the sweep's roofline divides by, as the microbenchmark's mode:
    2 = tagged 32-bit words (the layered sweep, and resident batches of at most two link
    candidates: one max and one min per candidate and cell), 0 = plain 32-bit words (max,
    compare, two selects), 1 = 64-bit words (a streaming sweep runs on those).  A batch
    whose instances take different words (a split resident sweep, or instances whose
    values need 64-bit words) is reported against the peak of its fastest words, an upper
    bound of the batch's effective peak: the fraction is then a lower bound."""
    if plan.get("sweep_variant") == 3:
        return 2   # layered: tagged 32-bit words, one max and one min per pair and cell
    if plan.get("sweep_variant") == 2:
        return 1
    return 2 if max(len(x.cand) for x in instances) <= 2 else 0


def stored_traffic(kernel, workload):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{kernel}@{workload}")
    if not d or d.get("src") != src_hash(kernel):
        return None
    return d.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_ms=20):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", f"-lms", str(period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(instances, seconds=12.0):
    """The oracle as it stands, one instance per host thread on all host cores, over a
    bounded sample of the batch: rounds of one instance per core (cycling through the
    batch) until `seconds` have passed, at least one round."""
    from oracle import oracle as O
    from concurrent.futures import ThreadPoolExecutor
    O.lib()
    cores = os.cpu_count() or 1
    n = min(cores, len(instances))
    t0 = time.perf_counter()
    done, relax, rounds = 0, 0, 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while True:
            batch = [instances[(done + q) % len(instances)] for q in range(n)]
            list(ex.map(oracle_solve, batch))
            done += n
            rounds += 1
            relax += sum(relaxations(x) for x in batch)
            if time.perf_counter() - t0 >= seconds:
                break
    dt = time.perf_counter() - t0
    return {"value": relax / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} instance solves ({rounds} round(s) of {n} in parallel, cycling through the "
                      f"{len(instances)}-instance batch), {dt:.1f} s",
            "solves_per_s": done / dt,
            "core_s_per_instance": dt * n / done}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def bench_config(workload, instances, chunk, relax_total, words, ws):
    """The `config` of the JSON line, the same for both arms."""
    return {"workload": workload, "batch_per_gpu": len(instances), "chunk": chunk,
            "relaxations_per_batch": relax_total, "cost_words_per_batch": words,
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)", "parallelism": f"replicas{ws}"}


def run_reference(args, workload, instances, relax_total):
    """The CPU oracle as the reference arm: each step solves a bounded sample."""
    rank, _, ws = dist_env()
    if rank != 0:
        return
    from oracle import oracle as O
    from concurrent.futures import ThreadPoolExecutor
    O.lib()
    cores = os.cpu_count() or 1
    per = [relaxations(x) for x in instances]
    # one step = as many instances as there are cores (cycling through the batch)
    n = min(cores, len(instances))
    times = []
    done_relax = 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        for step in range(args.warmup + args.steps):
            idx = [(step * n + q) % len(instances) for q in range(n)]
            t0 = time.perf_counter()
            list(ex.map(oracle_solve, [instances[q] for q in idx]))
            dt = time.perf_counter() - t0
            if step >= args.warmup:
                times.append(dt)
                done_relax += sum(per[q] for q in idx)
    total = sum(times)
    value = done_relax / total
    chunk = args.chunk if 0 < args.chunk < len(instances) else len(instances)
    words = sum(cost_words(x) for x in instances)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": bench_config(workload, instances, chunk, relax_total, words, ws),
            "reference": "CPU oracle (plain C), one instance per host thread; each step solves one instance "
                         "per host core, cycling through the batch",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} instance(s) per step over {args.steps} steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def rank_instances(workload_id: int, rank: int, batch: int = 0):
    """The batch one rank solves: its own B instances (seeds 1000 w + rank B + b), so
    ranks share nothing and need no exchange (the tiny workload is one fixed instance);
    `batch` > 0 takes the first `batch` of them."""
    B = synth.CONFIG_BATCH[workload_id]
    n = min(batch, B) if batch > 0 else B
    return synth.config_batch(workload_id, B=n, first=rank * B if workload_id != 1 else 0)


def job_totals(local_units: float, local_ms: float, dist=None, device=None):
    """Whole-job (units, ms): units summed over ranks, time the slowest rank's."""
    if dist is None:
        return local_units, local_ms
    import torch
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u.item()), float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 15 s of work)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--batch", type=int, default=0,
                    help="solve only the first N instances of the workload (0 = its whole batch); for "
                         "profiling captures on a small case")
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--sweep-variant", type=int, default=0, choices=[0, 1, 2, 3],
                    help="DP sweep variant: 0 = the library's choice, 1 = resident, 2 = streaming, "
                         "3 = layered (one launch per pipeline position)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = same as --steps (capped at 500)")
    ap.add_argument("--schedule", default="1f1b", choices=["1f1b", "gpipe"],
                    help="pipeline schedule of every instance (gpipe: all microbatches of a replica stashed)")
    ap.add_argument("--gpipe-microbatches", type=int, default=512,
                    help="microbatches per iteration under --schedule gpipe (4096 do not fit in memory)")
    ap.add_argument("--topology", default="tiers", choices=["tiers", "torus"],
                    help="torus: the dense workload's problems on a 4x4x4 torus of 64 chips, tiers = hop classes")
    ap.add_argument("--graph", default="chain", choices=["chain", "two-tower"],
                    help="two-tower: the dense workload's blocks as two 8-block encoder branches feeding a "
                         "16-block trunk, solved over the up-sets of that layer DAG")
    ap.add_argument("--cuda-graph", action="store_true",
                    help="capture one solve (all its kernels) in a CUDA graph and time its replays; the "
                         "dominant kernel's duration for the roofline then comes from the warm-up steps "
                         "(events cannot be read per replay)")
    ap.add_argument("--joint", action="store_true",
                    help="joint microbatch-size search: every problem solved with 1, 2, 4 and 8 samples "
                         "per microbatch, the best variant selected on the GPU")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {1: 2000, 2: 2000, 3: 500, 4: 500, 5: 20}[args.workload]
    if args.warmup is None:
        args.warmup = 3 if args.workload == 5 else 20
    if args.warmup < 3:
        args.warmup = 3

    rank, local_rank, ws = dist_env()
    workload = f"{synth.CONFIG_NAMES[args.workload]}"
    instances = rank_instances(args.workload, rank, args.batch)
    B = len(instances)
    if args.topology == "torus":
        if args.workload != 2:
            raise SystemExit("--topology torus applies to workload 2 (64 devices)")
        instances = [synth.torus_instance(rank * B + b) for b in range(B)]
        workload = synth.TORUS_NAME
    if args.graph == "two-tower":
        if args.workload != 2 or args.topology != "tiers":
            raise SystemExit("--graph two-tower applies to workload 2 on its tiers")
        instances = [synth.two_tower_instance(rank * B + b) for b in range(B)]
        workload = synth.TWO_TOWER_NAME
    if args.schedule == "gpipe":
        for x in instances:
            x.schedule, x.M = 1, max(args.gpipe_microbatches, x.Pmax)
        workload += f"-gpipe-M{args.gpipe_microbatches}"
    group = 1
    if args.joint:
        group = len(synth.MICROBATCH_SIZES)
        instances = synth.joint_batch(instances)
        B = len(instances)
        workload += "-joint-mbs" + "-".join(str(b) for b in synth.MICROBATCH_SIZES)
    relax_total = sum(relaxations(x) for x in instances)
    relax_s_total = sum(relaxations_with_strategies(x) for x in instances)

    if args.impl == "reference":
        run_reference(args, workload, instances, relax_total)
        return

    import torch
    from memory_aware_device_gb300 import nest
    torch.cuda.set_device(local_rank)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    dims = nest.make_dims(instances)
    solver = nest.Solver(dims, chunk=args.chunk, device=dev)
    records = nest.pack_records(instances, dims)
    solver.load(records)
    chunk = args.chunk if 0 < args.chunk < B else B
    nchunks = (B + chunk - 1) // chunk
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def make_opt(only=None):
        # events at every kernel boundary, or only around kernel `only` (the others keep
        # their programmatic dependent launches)
        ev = [torch.cuda.Event(enable_timing=True) if only is None or q % NEV in (only, only + 1) else None
              for q in range(NEV * nchunks)]
        return nest.options(chunk=args.chunk, events=ev, variant=args.sweep_variant), ev

    def kernel_ms(opts):   # average ms per step of each kernel, over all chunks
        out = {k: 0.0 for k in KERNELS}
        for _, ev in opts:
            for c in range(nchunks):
                for q, k in enumerate(KERNELS):
                    if ev[NEV * c + q] is not None and ev[NEV * c + q + 1] is not None:
                        out[k] += ev[NEV * c + q].elapsed_time(ev[NEV * c + q + 1])
        return {k: v / len(opts) for k, v in out.items()}

    best = torch.empty(B // group, dtype=torch.int32, device=dev)

    def step(opt, st=None):
        st = stream if st is None else st
        rc = nest.solve_raw(dims, solver.records, solver.costs, solver.plans, solver.workspace, st, opt)
        if rc:
            raise nest.NestError(rc)
        if group > 1:   # the joint search: best variant of every problem
            rc = nest.lib().nest_select_best(solver.costs.data_ptr(), B, group, best.data_ptr(),
                                             ctypes.c_void_p(st.cuda_stream))
            if rc:
                raise nest.NestError(rc, "nest_select_best")

    warm = [make_opt() for _ in range(args.warmup)]
    for o in warm:
        flush.zero_()
        step(o[0])
    torch.cuda.synchronize(dev)
    # correctness guard on the bench's own output: every instance solved or infeasible
    res = solver.results()
    assert all(r["status"] in (nest.SOLVED, nest.INFEASIBLE) for r in res), "solver reported errors"
    # the dominant kernel, from the warm-up steps; the timed steps record events around
    # it only (its live duration for the roofline)
    wk = kernel_ms(warm[len(warm) // 2:])
    dom = max(wk, key=wk.get)
    qdom = KERNELS.index(dom)

    graph = None
    if args.cuda_graph:
        # one solve captured once; each timed step replays it (the per-kernel events
        # cannot be recorded inside the graph, so the roofline uses the warm-up figures)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(nest.options(chunk=args.chunk, variant=args.sweep_variant), side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                step(nest.options(chunk=args.chunk, variant=args.sweep_variant), side)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)

    # one set of events per step, so nothing syncs inside the timed region
    opts = [make_opt(qdom) for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local_rank)
    time.sleep(0.05)
    for s in range(args.steps):
        flush.zero_()                      # L2 flush outside the timed events
        starts[s].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(opts[s][0])
        ends[s].record(stream)
    torch.cuda.synchronize(dev)
    dom_ms = kernel_ms(opts)[dom] if graph is None else wk[dom]
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    # per-kernel breakdown from a separate pass with events at every kernel boundary (a
    # second or two of steps)
    nbd = min(args.steps, 100, max(3, int(1500.0 / max(statistics.mean(step_ms), 1e-3))))
    bd = [make_opt() for _ in range(nbd)]
    for o in bd:
        flush.zero_()
        step(o[0])
    torch.cuda.synchronize(dev)
    kms = kernel_ms(bd)
    job_relax, total_ms = job_totals(relax_total, sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_relax / (ms_per_step * 1e-3)
    solves = B * ws / (ms_per_step * 1e-3)
    plan = nest.describe_launch(dims, nest.options(chunk=args.chunk, variant=args.sweep_variant))
    launches = (plan["kernels_per_chunk"] * plan["chunks"] + (1 if group > 1 else 0)) * args.steps

    # end to end through the host-buffer entry point: H2D records, solve, D2H results
    e2e_steps = args.e2e_steps or min(args.steps, 500)
    if group == 1:   # the device path's workspace is not needed any more
        solver.workspace = None
        torch.cuda.empty_cache()
    wsh = torch.empty(nest.workspace_size(dims, args.chunk, host=True), dtype=torch.uint8, device=dev)
    rec_pin = torch.from_numpy(records.ravel().copy()).pin_memory()
    costs_pin = torch.empty(B, dtype=torch.int64).pin_memory()
    plans_pin = torch.empty(B * nest.plan_bytes(dims), dtype=torch.uint8).pin_memory()
    hopt = nest.options(chunk=args.chunk, variant=args.sweep_variant)

    best_pin = torch.empty(max(B // group, 1), dtype=torch.int32).pin_memory()

    def host_step():
        import ctypes as C
        if group == 1:
            rc = nest.lib().nest_solve_host(C.byref(dims), rec_pin.data_ptr(), costs_pin.data_ptr(),
                                            plans_pin.data_ptr(), wsh.data_ptr(), wsh.numel(),
                                            C.c_void_p(stream.cuda_stream), C.byref(hopt))
            if rc:
                raise nest.NestError(rc, "nest_solve_host")
            return
        # the joint search through the device entry points: H2D records, solve, select,
        # D2H of the choices, t_batch values and plans
        solver.records.copy_(rec_pin, non_blocking=True)
        step(hopt)
        best_pin[:B // group].copy_(best, non_blocking=True)
        costs_pin.copy_(solver.costs, non_blocking=True)
        plans_pin.copy_(solver.plans, non_blocking=True)
        stream.synchronize()
    for _ in range(min(args.warmup, 3)):
        host_step()
    if dist is not None:
        dist.barrier()
    e2e_ms = []
    for _ in range(e2e_steps):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        host_step()
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    _, e2e_total = job_totals(relax_total, sum(e2e_ms), dist, dev)
    e2e_val = job_relax / (e2e_total / e2e_steps * 1e-3)
    assert nest.decode_plans(plans_pin.numpy(), dims) == res, "host entry point disagrees with device path"

    # roofline of the dominant kernel, on its duration inside the timed steps
    peaks = load_peaks()
    words = sum(cost_words(x) for x in instances)
    if dom == "dp_sweep":
        mhz = (clk or {}).get("sm_mhz") or peaks["sm_max_mhz"]
        derived = alu_peak_relax_per_s(peaks["sm_max_mhz"]) / 1e9
        achieved = relax_total / (dom_ms * 1e-3) / 1e9
        # the peak is measured on the op mix the sweep issues
        mode = relax_peak_mode(instances, plan)
        meas = measured_relax_peak(mode)
        meas_plain = measured_relax_peak(0) if mode else meas
        # without the microbenchmark: INT32 lanes x clock / the mix's operations per relaxation
        ops = {2: 2, 0: 4, 1: OPS_PER_RELAX}[mode]
        peak = meas / 1e9 if meas else SMS * INT32_LANES * peaks["sm_max_mhz"] * 1e6 / ops / 1e9
        mix = ("tagged 32-bit words (one max and one min per candidate and cell)" if mode == 2 else
               "64-bit words (max, compare, two selects per candidate and cell)" if mode == 1 else
               "32-bit words (max, compare, two selects per candidate and cell)")
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Grelax/s",
                "frac": achieved / peak, "traffic": stored_traffic(dom, workload), "kernel": dom,
                "peak_source": (f"measured: register-only microbenchmark of the relaxation arithmetic on {mix}; "
                                "4 independent chains per thread, every SM full - the words this batch's sweep "
                                "runs on"
                                if meas else
                                f"derived: {SMS} SMs x {INT32_LANES} INT32 lanes x {peaks['sm_max_mhz']:.0f} MHz"
                                f" / {ops} ops per relaxation ({mix})"),
                "peak_plain_32bit": meas_plain / 1e9 if meas_plain else None,
                "derived_64bit_peak": derived, "sm_mhz_seen": mhz}
    else:
        # the per-position loads table is what the stage-loads kernel must write
        loads_bytes = sum(8 * x.Pmax * state_pairs(x) * (x.D // x.unit).bit_length() for x in instances)
        algo = {"stage_loads": loads_bytes, "prep": 0, "backtrack": 0}[dom]
        achieved = algo / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": stored_traffic(dom, workload),
                "kernel": dom, "peak_source": f"{peaks['source']} hbm_gbs"}
    # the stage-loads kernel (cost build + strategy reduction) against HBM, on the cost
    # builder's algorithmic bytes: 8 bytes per (stage, width, strategy) cost word written.
    # The fused kernel reduces the words in shared memory instead of writing them (and of
    # reading them back for the strategy reduction); its bound is integer arithmetic
    k1_bytes = 8 * words
    roof_loads = {"bound": "hbm", "kernel": "stage_loads", "achieved": k1_bytes / (kms["stage_loads"] * 1e-3) / 1e9,
                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "frac": k1_bytes / (kms["stage_loads"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "traffic": stored_traffic("stage_loads", workload),
                  "cost_words_per_s": words / (kms["stage_loads"] * 1e-3),
                  "note": "achieved = 8 B per cost word (the cost tensor the fused kernel never writes) over "
                          "its time; integer-ALU bound: exact 64-bit collective prices, shared per strategy "
                          "group"}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(instances, args.cpu_seconds)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
                "config": bench_config(workload, instances, chunk, relax_total, words, ws),
                "launch": plan,
                "solves_per_s": solves,
                "relaxations_jmsc_per_s": job_relax / relax_total * relax_s_total / (ms_per_step * 1e-3),
                "relaxations_jmsc_note": "the (j, m, s, c') count of the recurrence with the strategy axis, "
                                         "per second of the whole step",
                **({"problems_per_s": solves / group, "variants_per_problem": group} if group > 1 else {}),
                "kernel_ms_per_step": kms,
                "launch_mode": ("CUDA graph: each timed step replays one captured solve" if graph is not None
                                else "direct launches, events around the dominant kernel"),
                "kernel_ms_note": "separate pass, events at every kernel boundary (no launch overlap)",
                "roofline": roof, "roofline_stage_loads": roof_loads, "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": int(records.nbytes),
                        "d2h_bytes_per_step": int(B * nest.plan_bytes(dims) + (8 * B + 4 * (B // group) if group > 1 else 0)),
                        "ms_per_step": e2e_total / e2e_steps},
                "gpu_launches": launches, "clocks": clk}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
