"""Python binding of libnest (include/nest.h): argument marshalling only.

Every step of the solve runs in the library's CUDA kernels; this module packs
instances into the record layout the library reports, passes device pointers
and a stream, and decodes the plan records.  PyTorch supplies device memory and
streams.  There is no CPU fallback: if libnest.so is missing, loading fails.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnest.so")

NEST_OK, NEST_E_INVALID, NEST_E_LIMITS, NEST_E_WORKSPACE, NEST_E_CUDA, NEST_E_TIMEOUT = 0, -1, -2, -3, -4, -5
SOLVED, INFEASIBLE, BAD_INPUT, TIMED_OUT = 0, 1, 2, 3
CAP = (1 << 40) - 1
ERRORS = {NEST_E_INVALID: "invalid argument", NEST_E_LIMITS: "batch dimensions beyond the limits",
          NEST_E_WORKSPACE: "workspace too small or misaligned", NEST_E_CUDA: "CUDA call failed",
          NEST_E_TIMEOUT: "a device wait gave up"}

# Every function declared in include/nest.h.
EXPORTS = ("nest_record_layout", "nest_plan_bytes", "nest_workspace_size", "nest_workspace_size_costs",
           "nest_workspace_layout", "nest_solve", "nest_workspace_size_host", "nest_solve_host",
           "nest_select_best", "nest_solve_static", "nest_describe_launch")
KEEP_COSTS = 1   # NEST_KEEP_COSTS
STATIC_SCRATCH_BYTES = 64 << 20   # NEST_STATIC_SCRATCH_BYTES


class NestError(RuntimeError):
    def __init__(self, rc: int, what: str = "nest_solve"):
        super().__init__(f"{what} returned {rc}: {ERRORS.get(rc, 'unknown error')}")
        self.rc = rc


class Dims(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("B", "Lmax", "Tmax", "Cmax", "Smax", "Pcap", "Dumax", "Vmax")]


class Layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("record_bytes", "fl", "pd", "pe", "ao", "aw", "a2a", "moe",
                                         "G", "bw", "lat", "cand", "strat", "succ")]


class WsLayout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("loads", "dpv", "dpa", "cost", "total", "total_costs")] + \
               [(n, C.c_int32) for n in ("NP", "Kmax", "Kpad", "Spad", "Dpad", "chunk", "N", "reserved")]


class Options(C.Structure):
    _fields_ = [("chunk", C.c_int32), ("sweep_cluster", C.c_int32), ("sweep_jsplit", C.c_int32),
                ("sweep_variant", C.c_int32), ("spin_limit", C.c_int64), ("events", C.c_void_p),
                ("flags", C.c_uint32), ("reserved", C.c_int32)]


class LaunchDesc(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("chunks", "kernels_per_chunk", "sweep_variant", "sweep_cluster",
                                         "sweep_jsplit", "sweep_threads", "sweep_split", "wide_variant",
                                         "wide_cluster", "wide_jsplit", "wide_threads", "reserved")]


HEADER_DT = np.dtype([("L", "<i4"), ("D", "<i4"), ("unit", "<i4"), ("T", "<i4"), ("C", "<i4"),
                      ("S", "<i4"), ("Pmax", "<i4"), ("schedule", "<i4"), ("R", "<i8"), ("M", "<i8"),
                      ("budget", "<i8"), ("opt_factor", "<i8"), ("graph", "<i4"), ("reserved", "<i4")])
PLAN_HDR_DT = np.dtype([("status", "<i4"), ("n_stages", "<i4"), ("t_batch", "<i8"), ("bottleneck", "<i8")])
STAGE_DT = np.dtype([("i", "<i2"), ("j", "<i2"), ("s", "<i2"), ("c_next", "i1"), ("reserved", "i1"),
                     ("k", "<i4"), ("reserved2", "<i4"), ("layers", "<u8")])

_lib = None


def lib():
    """Load libnest.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(the solver has no CPU fallback)")
        L = C.CDLL(LIB_PATH)
        P = C.POINTER
        L.nest_record_layout.argtypes = [P(Dims), P(Layout)]
        L.nest_plan_bytes.argtypes = [P(Dims)]
        L.nest_plan_bytes.restype = C.c_size_t
        L.nest_workspace_size.argtypes = [P(Dims), C.c_int32]
        L.nest_workspace_size.restype = C.c_size_t
        L.nest_workspace_size_costs.argtypes = [P(Dims), C.c_int32]
        L.nest_workspace_size_costs.restype = C.c_size_t
        L.nest_workspace_size_host.argtypes = [P(Dims), C.c_int32]
        L.nest_workspace_size_host.restype = C.c_size_t
        L.nest_workspace_layout.argtypes = [P(Dims), C.c_int32, P(WsLayout)]
        L.nest_solve.argtypes = [P(Dims), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                 C.c_void_p, P(Options)]
        L.nest_solve_host.argtypes = [P(Dims), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                      C.c_void_p, P(Options)]
        L.nest_solve_static.argtypes = [P(Dims), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, P(Options)]
        L.nest_select_best.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
        L.nest_describe_launch.argtypes = [P(Dims), P(Options), P(LaunchDesc)]
        _lib = L
    return _lib


# ---------------------------------------------------------------------------------
# Geometry and packing
# ---------------------------------------------------------------------------------

def upset_count(succ, limit: int = 256) -> int:
    """Number of up-sets of the layer DAG given by successor masks (the empty set
    included), counted up to `limit` + 1: sizes the batch (nest_dims.Vmax); the
    library enumerates and checks the states itself."""
    L = len(succ)
    sc = [int(v) for v in succ]
    n = 0
    stack = [(L - 1, 0)]          # decide layers from the last one down
    while stack and n <= limit:
        l, D = stack.pop()
        if l < 0:
            n += 1
            continue
        stack.append((l - 1, D))
        if sc[l] & ~D == 0:
            stack.append((l - 1, D | (1 << l)))
    return n


def make_dims(instances: Sequence, Pcap: int | None = None, Dumax: int | None = None,
              Vmax: int | None = None) -> Dims:
    """Batch dims covering `instances`; an instance with a `succ` attribute (not None)
    is a graph instance, and Vmax defaults to its largest up-set count less one."""
    if Vmax is None:
        Vmax = max([upset_count(x.succ) - 1 for x in instances if getattr(x, "succ", None) is not None],
                   default=0)
    return Dims(B=len(instances), Lmax=max(int(x.L) for x in instances),
                Tmax=max(len(x.tierG) for x in instances), Cmax=max(len(x.cand) for x in instances),
                Smax=max(len(x.strat) for x in instances),
                Pcap=Pcap or max(int(x.Pmax) for x in instances),
                Dumax=Dumax or max(int(x.D) // int(x.unit) for x in instances), Vmax=Vmax)


def record_layout(dims: Dims) -> Layout:
    out = Layout()
    rc = lib().nest_record_layout(C.byref(dims), C.byref(out))
    if rc:
        raise NestError(rc, "nest_record_layout")
    return out


def plan_bytes(dims: Dims) -> int:
    return int(lib().nest_plan_bytes(C.byref(dims)))


def workspace_size(dims: Dims, chunk: int = 0, host: bool = False, keep_costs: bool = False) -> int:
    f = lib().nest_workspace_size_host if host else \
        lib().nest_workspace_size_costs if keep_costs else lib().nest_workspace_size
    return int(f(C.byref(dims), chunk))


def workspace_layout(dims: Dims, chunk: int = 0) -> WsLayout:
    out = WsLayout()
    rc = lib().nest_workspace_layout(C.byref(dims), chunk, C.byref(out))
    if rc:
        raise NestError(rc, "nest_workspace_layout")
    return out


def describe_launch(dims: Dims, opt: Options | None = None) -> dict:
    """nest_describe_launch: the passes, kernels per pass and DP-sweep shape of a solve."""
    out = LaunchDesc()
    rc = lib().nest_describe_launch(C.byref(dims), C.byref(opt) if opt is not None else None, C.byref(out))
    if rc:
        raise NestError(rc, "nest_describe_launch")
    return {n: int(getattr(out, n)) for n, _ in LaunchDesc._fields_ if n != "reserved"}


def pack_records(instances: Sequence, dims: Dims, out: np.ndarray | None = None) -> np.ndarray:
    """Instance records in the library's layout: uint8 [B, record_bytes]."""
    lay = record_layout(dims)
    rb = lay.record_bytes
    buf = out if out is not None else np.zeros((len(instances), rb), dtype=np.uint8)
    buf[...] = 0
    for b, x in enumerate(instances):
        row = buf[b]
        h = np.zeros(1, HEADER_DT)
        h["L"], h["D"], h["unit"], h["T"], h["C"], h["S"], h["Pmax"] = (
            x.L, x.D, x.unit, len(x.tierG), len(x.cand), len(x.strat), x.Pmax)
        h["R"], h["M"], h["budget"], h["opt_factor"] = x.R, x.M, x.budget, x.opt_factor
        h["schedule"] = int(getattr(x, "schedule", 0))
        succ = getattr(x, "succ", None)
        h["graph"] = 0 if succ is None else 1
        row[:HEADER_DT.itemsize] = h.view(np.uint8)

        def put(off, arr, dt):
            a = np.ascontiguousarray(np.asarray(arr, dtype=dt)).view(np.uint8).ravel()
            row[off:off + a.size] = a
        for f in ("fl", "pd", "pe", "ao", "aw", "a2a"):
            put(getattr(lay, f), getattr(x, f), "<i8")
        put(lay.moe, x.moe, np.uint8)
        put(lay.G, x.tierG, "<i8")
        put(lay.bw, x.tierBw, "<i8")
        put(lay.lat, x.tierLat, "<i8")
        put(lay.cand, x.cand, "<i4")
        st = np.zeros((len(x.strat), 8), dtype="<i2")
        st[:, :5] = np.asarray(x.strat, dtype=np.int16).reshape(-1, 5)
        put(lay.strat, st, "<i2")
        if succ is not None:
            put(lay.succ, succ, "<u8")
    return buf


def decode_plans(raw: np.ndarray, dims: Dims) -> List[dict]:
    """Plan records -> [{status, t_batch, bottleneck, plan: [(i, j, k, s, c_next)],
    layers: [layer mask of each stage]}]."""
    pb = plan_bytes(dims)
    raw = np.ascontiguousarray(raw).view(np.uint8).reshape(dims.B, pb)
    out = []
    for b in range(dims.B):
        h = raw[b, :PLAN_HDR_DT.itemsize].view(PLAN_HDR_DT)[0]
        n = int(h["n_stages"])
        st = raw[b, PLAN_HDR_DT.itemsize:PLAN_HDR_DT.itemsize + n * STAGE_DT.itemsize].view(STAGE_DT)
        out.append({"status": int(h["status"]), "t_batch": int(h["t_batch"]),
                    "bottleneck": int(h["bottleneck"]),
                    "plan": [(int(s["i"]), int(s["j"]), int(s["k"]), int(s["s"]), int(s["c_next"]))
                             for s in st],
                    "layers": [int(s["layers"]) for s in st]})
    return out


def options(chunk=0, cluster=0, jsplit=0, spin_limit=0, events=None, variant=0, keep_costs=False) -> Options:
    o = Options(chunk=chunk, sweep_cluster=cluster, sweep_jsplit=jsplit, sweep_variant=variant,
                spin_limit=spin_limit, events=None, flags=KEEP_COSTS if keep_costs else 0)
    if events is not None:   # torch.cuda.Event entries; None entries are not recorded
        for e in events:
            if e is not None and not e.cuda_event:   # torch creates the CUDA event lazily
                e.record()
        arr = (C.c_void_p * len(events))(*[e.cuda_event if e is not None else None for e in events])
        o._events_keep = (arr, list(events))   # the CUDA events live as long as the options
        o.events = C.cast(arr, C.c_void_p)
    return o


# ---------------------------------------------------------------------------------
# Calls
# ---------------------------------------------------------------------------------

def solve_raw(dims: Dims, records, costs, plans, workspace, stream=None, opt: Options | None = None) -> int:
    """nest_solve on torch CUDA tensors (uint8 records/plans/workspace, int64 costs)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return lib().nest_solve(C.byref(dims), records.data_ptr(), costs.data_ptr(), plans.data_ptr(),
                            workspace.data_ptr(), workspace.numel(), C.c_void_p(stream.cuda_stream),
                            C.byref(opt) if opt is not None else None)


def solve_host_raw(dims: Dims, records_host: np.ndarray, costs_host: np.ndarray, plans_host: np.ndarray,
                   workspace, stream=None, opt: Options | None = None) -> int:
    """nest_solve_host: HOST records in, HOST costs and plans out (synchronous)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return lib().nest_solve_host(C.byref(dims), records_host.ctypes.data, costs_host.ctypes.data,
                                 plans_host.ctypes.data, workspace.data_ptr(), workspace.numel(),
                                 C.c_void_p(stream.cuda_stream), C.byref(opt) if opt is not None else None)


class Solver:
    """Owns device buffers (via torch) for repeated solves of batches with fixed dims."""

    def __init__(self, dims: Dims, chunk: int = 0, device="cuda", host_io: bool = False, keep_costs: bool = False):
        import torch
        self.dims = dims
        self.chunk = chunk
        self.device = torch.device(device)
        self.layout = record_layout(dims)
        self.pb = plan_bytes(dims)
        B = dims.B
        self.records = torch.empty(B * self.layout.record_bytes, dtype=torch.uint8, device=self.device)
        self.costs = torch.empty(B, dtype=torch.int64, device=self.device)
        self.plans = torch.empty(B * self.pb, dtype=torch.uint8, device=self.device)
        ws = workspace_size(dims, chunk, host=host_io, keep_costs=keep_costs)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)

    def load(self, records_np: np.ndarray):
        import torch
        self.records.copy_(torch.from_numpy(np.ascontiguousarray(records_np).ravel()))

    def run(self, stream=None, opt: Options | None = None):
        rc = solve_raw(self.dims, self.records, self.costs, self.plans, self.workspace, stream, opt)
        if rc:
            raise NestError(rc)

    def results(self) -> List[dict]:
        return decode_plans(self.plans.cpu().numpy(), self.dims)

    def capture(self, opt: Options | None = None):
        """One solve of the loaded records captured in a CUDA graph (nest_solve only enqueues
        kernels, so it captures as is); graph.replay() re-runs it on the current stream."""
        import torch
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            self.run(stream=side, opt=opt)   # launch attributes set outside the capture
            with torch.cuda.graph(graph, stream=side):
                self.run(stream=side, opt=opt)
        torch.cuda.current_stream(self.device).wait_stream(side)
        return graph


def select_best(costs, group: int, stream=None):
    """nest_select_best on a torch int64 CUDA tensor of t_batch values: the best index
    within each group of `group` consecutive instances (int32 tensor, -1 = none)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(costs.device)
    best = torch.empty(costs.numel() // group if group > 0 else 0, dtype=torch.int32, device=costs.device)
    rc = lib().nest_select_best(costs.data_ptr(), costs.numel(), group, best.data_ptr(),
                                C.c_void_p(stream.cuda_stream))
    if rc:
        raise NestError(rc, "nest_select_best")
    return best


def solve_instances(instances: Sequence, device="cuda", **opt_kw) -> List[dict]:
    """Convenience: pack, solve on the GPU, decode."""
    import torch
    dims = make_dims(instances)
    s = Solver(dims, chunk=opt_kw.get("chunk", 0), device=device)
    s.load(pack_records(instances, dims))
    s.run(opt=options(**opt_kw))
    torch.cuda.synchronize(s.device)
    return s.results()
