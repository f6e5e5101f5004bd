"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/nest.h declares, reports consistent layouts, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from memory_aware_device_gb300 import build as nbuild
from memory_aware_device_gb300 import nest, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    nbuild.build()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "nest.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(nest_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(nest.EXPORTS)
    L = C.CDLL(nest.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_no_dynamic_allocation_symbols_in_api_source():
    src = open(os.path.join(ROOT, "memory_aware_device_gb300", "csrc", "nest_api.cu")).read()
    for bad in ("cudaMalloc", "cudaFree", "malloc(", "new "):
        assert bad not in src


def test_record_layout_is_aligned():
    dims = nest.make_dims(synth.config_batch(2))
    lay = nest.record_layout(dims)
    assert lay.record_bytes % 256 == 0
    offs = [lay.fl, lay.pd, lay.pe, lay.ao, lay.aw, lay.a2a, lay.moe, lay.G, lay.bw, lay.lat, lay.cand, lay.strat]
    assert offs == sorted(offs) and all(o % 16 == 0 for o in offs)
    assert lay.fl >= 64 and lay.strat + 16 * dims.Smax <= lay.record_bytes


def test_pack_roundtrip():
    insts = synth.config_batch(4, B=3)
    dims = nest.make_dims(insts)
    lay = nest.record_layout(dims)
    rec = nest.pack_records(insts, dims)
    for b, x in enumerate(insts):
        h = rec[b, :nest.HEADER_DT.itemsize].view(nest.HEADER_DT)[0]
        assert (h["L"], h["D"], h["unit"], h["S"], h["budget"]) == (x.L, x.D, x.unit, len(x.strat), x.budget)
        fl = rec[b, lay.fl:lay.fl + 8 * x.L].view("<i8")
        assert (fl == x.fl).all()
        st = rec[b, lay.strat:lay.strat + 16 * len(x.strat)].view("<i2").reshape(-1, 8)
        assert (st[:, :5] == x.strat).all() and (st[:, 5:] == 0).all()


@pytest.mark.parametrize("field,value", [("Lmax", 256), ("Lmax", 0), ("Tmax", 9), ("Cmax", 16),
                                         ("Smax", 4096), ("Pcap", 32), ("Dumax", 513), ("Dumax", 0),
                                         ("Vmax", 256), ("Vmax", -1)])
def test_limits_rejected_on_host(field, value):
    dims = nest.make_dims(synth.config_batch(2, B=2))
    setattr(dims, field, value)
    assert nest.workspace_size(dims) == 0
    assert nest.plan_bytes(dims) == 0
    rc = nest.lib().nest_solve(C.byref(dims), None, None, None, None, 0, None, None)
    assert rc == nest.NEST_E_LIMITS


def test_largest_dims_accepted():
    dims = nest.Dims(B=1, Lmax=255, Tmax=8, Cmax=15, Smax=4095, Pcap=31, Dumax=512, Vmax=255)
    assert nest.workspace_size(dims) > 0 and nest.plan_bytes(dims) == 24 + 24 * 31
    assert nest.STAGE_DT.itemsize == 24 and nest.HEADER_DT.itemsize == 72


def test_state_dimension_follows_the_larger_of_layers_and_up_sets():
    base = dict(B=1, Lmax=32, Tmax=3, Cmax=2, Smax=12, Pcap=16, Dumax=64)
    chain = nest.workspace_layout(nest.Dims(**base, Vmax=0))
    graph = nest.workspace_layout(nest.Dims(**base, Vmax=96))
    assert (chain.N, chain.NP) == (32, 32 * 33 // 2)
    assert (graph.N, graph.NP) == (96, 96 * 97 // 2)
    assert nest.workspace_layout(nest.Dims(**base, Vmax=20)).N == 32


@pytest.mark.parametrize("seed", range(30))
def test_upset_count_sizes_the_batch(seed):
    O = pytest.importorskip("oracle.oracle")
    x = synth.random_tiny(seed, Lmax=8)
    succ = synth.random_dag(seed, x.L, (0.1, 0.4, 0.8)[seed % 3])
    assert nest.upset_count(succ) == len(O.lattice_states(x, succ))
    assert nest.upset_count(synth.two_tower_succ()) == 97
    assert nest.upset_count(synth.chain_succ(12)) == 13


def test_bad_arguments_rejected_before_any_launch():
    dims = nest.make_dims(synth.config_batch(2, B=2))
    L = nest.lib()
    assert L.nest_solve(None, None, None, None, None, 0, None, None) == nest.NEST_E_INVALID
    assert L.nest_solve(C.byref(dims), None, None, None, None, 0, None, None) == nest.NEST_E_INVALID
    fake = 1 << 20   # never dereferenced: the size check fails first
    assert L.nest_solve(C.byref(dims), fake, fake, fake, fake, 16, None, None) == nest.NEST_E_WORKSPACE
    assert L.nest_solve(C.byref(dims), fake + 8, fake, fake, fake, 1 << 40, None, None) == nest.NEST_E_WORKSPACE
    neg = nest.Dims(B=-1, Lmax=4, Tmax=1, Cmax=1, Smax=1, Pcap=1, Dumax=1)
    assert L.nest_solve(C.byref(neg), None, None, None, None, 0, None, None) == nest.NEST_E_INVALID
    zero = nest.Dims(B=0, Lmax=4, Tmax=1, Cmax=1, Smax=1, Pcap=1, Dumax=1)
    assert L.nest_solve(C.byref(zero), None, None, None, None, 0, None, None) == nest.NEST_OK
    assert L.nest_solve_host(C.byref(zero), None, None, None, None, 0, None, None) == nest.NEST_OK


def test_select_best_rejects_bad_groups_before_any_launch():
    L = nest.lib()
    fake = 1 << 20   # never dereferenced: the checks fail first
    assert L.nest_select_best(fake, 8, 0, fake, None) == nest.NEST_E_INVALID
    assert L.nest_select_best(fake, 10, 4, fake, None) == nest.NEST_E_INVALID
    assert L.nest_select_best(fake, -4, 4, fake, None) == nest.NEST_E_INVALID
    assert L.nest_select_best(None, 0, 4, None, None) == nest.NEST_OK
    assert L.nest_select_best(None, 8, 4, fake, None) == nest.NEST_E_INVALID


def test_workspace_grows_with_chunk_and_matches_layout():
    dims = nest.make_dims(synth.config_batch(3, B=8))
    a, b = nest.workspace_size(dims, 2), nest.workspace_size(dims, 8)
    assert 0 < a < b
    lay = nest.workspace_layout(dims, 8)
    assert lay.total == b and lay.chunk == 8
    assert lay.loads < lay.dpv < lay.dpa < lay.total == lay.cost < lay.total_costs
    assert lay.total_costs == nest.workspace_size(dims, 8, keep_costs=True)
    assert lay.NP == 96 * 97 // 2 and lay.Kmax == 8 and lay.Dpad == 132 and lay.Spad == 36
    assert nest.workspace_size(dims, 0) == b and nest.workspace_size(dims, 99) == b
    assert nest.workspace_size(dims, 8, host=True) > b


def test_cost_tensor_sizes_match_workload_table():
    # stage-cost words per instance: L(L+1)/2 pairs x widths x strategies
    for cfg, words in ((1, 1152), (2, 44352), (3, 1340928), (4, 460992), (5, 55480320)):
        x = synth.config_instance(cfg, 0)
        K = (x.D // x.unit).bit_length()
        assert x.L * (x.L + 1) // 2 * K * len(x.strat) == words


def test_describe_launch_without_a_device():
    # no GPU here: no resident shape can be sized, so the shape falls back to the layered
    # sweep (position 1, a launch per tag mode for each later position, the streaming
    # launch for the instances beyond its words), followed by the backtrack
    dims = nest.make_dims(synth.config_batch(2, B=4))
    d = nest.describe_launch(dims)
    assert d["chunks"] == 1 and d["sweep_variant"] in (1, 2, 3)
    per = {1: 3 + d["sweep_split"], 2: 4 + d["sweep_split"], 3: 2 + 1 + 2 * (dims.Pcap - 1) + 1 + 1}
    assert d["kernels_per_chunk"] == per[d["sweep_variant"]]
    for v in (2, 3):
        assert nest.describe_launch(dims, nest.options(variant=v))["sweep_variant"] == v
    with pytest.raises(nest.NestError):
        nest.describe_launch(dims, nest.options(variant=4))
    assert nest.describe_launch(dims, nest.options(chunk=3))["chunks"] == 2
    bad = nest.Dims(B=1, Lmax=256, Tmax=1, Cmax=1, Smax=1, Pcap=1, Dumax=1)
    with pytest.raises(nest.NestError):
        nest.describe_launch(bad)
    assert nest.lib().nest_describe_launch(C.byref(dims), None, None) == nest.NEST_E_INVALID


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    # there is no CPU fallback: with libnest.so absent, loading raises instead of solving
    monkeypatch.setattr(nest, "_lib", None)
    monkeypatch.setattr(nest, "LIB_PATH", str(tmp_path / "libnest.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        nest.lib()
    with pytest.raises(RuntimeError):
        nest.make_dims(synth.config_batch(1)) and nest.record_layout(nest.make_dims(synth.config_batch(1)))
