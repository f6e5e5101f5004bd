"""The entry point that allocates nothing (nest_solve_static), called through the C ABI.

It serves callers that cannot allocate device memory (a process whose allocator owns
all device memory, a plug-in whose host forbids device allocations, code that must
not stall on cudaMalloc / cudaFree): its scratch is a fixed array inside the
library.  Its results must equal those of nest_solve with a caller-provided
workspace, on two calls in a row (the array keeps the previous call's contents).
This file is collected last, so that a failure here comes after every other test.
"""
import ctypes as C

import numpy as np
import pytest

from memory_aware_device_gb300 import build as nbuild
from memory_aware_device_gb300 import nest, synth

pytestmark = pytest.mark.gpu


def _reference(insts, chunk=0):
    """nest_solve with a caller-provided workspace that starts full of 0xFF bytes."""
    import torch
    dims = nest.make_dims(insts)
    s = nest.Solver(dims, chunk=chunk)
    s.workspace.fill_(0xFF)
    s.load(nest.pack_records(insts, dims))
    s.run(opt=nest.options(chunk=chunk))
    torch.cuda.synchronize()
    return s.costs.cpu().numpy().copy(), s.plans.cpu().numpy().copy()


def _static(insts, opt=None):
    """One nest_solve_static call; returns (rc, costs, plans)."""
    import torch
    dims = nest.make_dims(insts)
    records = torch.from_numpy(nest.pack_records(insts, dims).ravel()).cuda()
    costs = torch.full((len(insts),), -7, dtype=torch.int64, device="cuda")
    plans = torch.zeros(len(insts) * nest.plan_bytes(dims), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    rc = nest.lib().nest_solve_static(C.byref(dims), records.data_ptr(), costs.data_ptr(), plans.data_ptr(),
                                      C.c_void_p(stream.cuda_stream), C.byref(opt) if opt is not None else None)
    torch.cuda.synchronize()
    return rc, costs.cpu().numpy(), plans.cpu().numpy()


# before each case the array holds another workload's solve (another one of the list)
CASES = [(2, 16), (1, 1), (4, 8)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_workspace_entry_point(case):
    import torch
    assert torch.cuda.is_available(), "GPU test"
    nbuild.build()
    workload, B = CASES[case]
    other_w, other_B = CASES[(case + 1) % len(CASES)]
    assert _static(synth.config_batch(other_w, B=other_B))[0] == nest.NEST_OK
    insts = synth.config_batch(workload, B=B)
    dims = nest.make_dims(insts)
    assert 0 < nest.workspace_size(dims) <= nest.STATIC_SCRATCH_BYTES
    want_costs, want_plans = _reference(insts)
    records = torch.from_numpy(nest.pack_records(insts, dims).ravel()).cuda()
    stream = torch.cuda.current_stream()
    for call in range(2):
        costs = torch.full((B,), -7, dtype=torch.int64, device="cuda")
        plans = torch.zeros(B * nest.plan_bytes(dims), dtype=torch.uint8, device="cuda")
        rc = nest.lib().nest_solve_static(C.byref(dims), records.data_ptr(), costs.data_ptr(), plans.data_ptr(),
                                          C.c_void_p(stream.cuda_stream), None)
        assert rc == nest.NEST_OK, (call, rc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(costs.cpu().numpy(), want_costs)
        got = nest.decode_plans(plans.cpu().numpy(), dims)
        assert got == nest.decode_plans(want_plans, dims)
        assert all(r["status"] == nest.SOLVED for r in got)


def test_static_scratch_rejects_batches_beyond_its_size():
    import torch
    nbuild.build()
    insts = synth.config_batch(3, B=8)   # needs about 190 MB of scratch
    dims = nest.make_dims(insts)
    assert nest.workspace_size(dims) > nest.STATIC_SCRATCH_BYTES
    records = torch.from_numpy(nest.pack_records(insts, dims).ravel()).cuda()
    costs = torch.zeros(8, dtype=torch.int64, device="cuda")
    plans = torch.zeros(8 * nest.plan_bytes(dims), dtype=torch.uint8, device="cuda")
    rc = nest.lib().nest_solve_static(C.byref(dims), records.data_ptr(), costs.data_ptr(), plans.data_ptr(),
                                      None, None)
    assert rc == nest.NEST_E_WORKSPACE
    # a chunk small enough for the array is accepted, and solves as nest_solve does with
    # the same chunk
    rc, got_costs, got_plans = _static(insts, nest.options(chunk=2))
    assert rc == nest.NEST_OK
    want_costs, want_plans = _reference(insts, chunk=2)
    np.testing.assert_array_equal(got_costs, want_costs)
    assert nest.decode_plans(got_plans, dims) == nest.decode_plans(want_plans, dims)


def test_static_scratch_refuses_kept_costs():
    # the stage-cost tensor would be written into the library's array, out of reach
    nbuild.build()
    insts = synth.config_batch(2, B=2)
    assert _static(insts, nest.options(keep_costs=True))[0] == nest.NEST_E_INVALID
    assert _static(insts)[0] == nest.NEST_OK
