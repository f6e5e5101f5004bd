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


def _reference(insts):
    import torch
    dims = nest.make_dims(insts)
    s = nest.Solver(dims)
    s.load(nest.pack_records(insts, dims))
    s.run()
    torch.cuda.synchronize()
    return s.costs.cpu().numpy().copy(), s.plans.cpu().numpy().copy()


@pytest.mark.parametrize("workload,B", [(2, 16), (1, 1), (4, 8)])
def test_static_scratch_matches_workspace_entry_point(workload, B):
    import torch
    assert torch.cuda.is_available(), "GPU test"
    nbuild.build()
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
    # a chunk small enough for the array is accepted
    opt = nest.options(chunk=2)
    rc = nest.lib().nest_solve_static(C.byref(dims), records.data_ptr(), costs.data_ptr(), plans.data_ptr(),
                                      None, C.byref(opt))
    assert rc == nest.NEST_OK
    torch.cuda.synchronize()
    assert all(r["status"] in (nest.SOLVED, nest.INFEASIBLE) for r in nest.decode_plans(plans.cpu().numpy(), dims))
