// nest_solve_static: the same solve as nest_solve, for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a serving or scheduling
// process that has already handed all device memory to its own pool (a further
// cudaMalloc fails, or fragments the pool it manages), a plug-in that runs inside a
// host application which forbids device allocations in its callbacks, and code that
// must not stall on the device-wide synchronisation that cudaMalloc and cudaFree can
// cause.  For them the scratch memory of the solve (the workspace of nest_solve)
// lives in a fixed array inside the library instead of a caller-provided buffer.
//
// The array is NEST_STATIC_SCRATCH_BYTES long and every GPU that loads the library
// holds it until the process exits.  Its device address is looked up with that device
// current (cudaGetSymbolAddress) on every call made outside a stream capture, so it
// stays right after a device reset; a call made while its stream is being captured
// uses the address of the last call outside a capture on that device, so make one call
// before capturing.  Every call shares the array and it keeps the last call's
// contents; nothing in it needs clearing, because the solve writes every scratch word
// before it reads it.  Calls whose work overlaps on the GPU (two streams, or two host
// threads) race on the array and must be serialised by the caller.  NEST_KEEP_COSTS is
// refused: the stage-cost tensor would land in the array, where the caller cannot read
// it.
#include <cuda_runtime.h>

#include <mutex>

#include "nest_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[NEST_STATIC_SCRATCH_BYTES];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per device

// Device address of the scratch array on the current device: looked up again unless
// `stream` is being captured (then the last address looked up on this device).
int scratch_address(void *stream, void **out) {
    int dev = 0;
    if (int rc = nest::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
    if (dev < 0 || dev >= kMaxDevices) return NEST_E_INVALID;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (int rc = nest::cuda_status(cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap),
                                   "cudaStreamIsCapturing"))
        return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (cap == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
        if (cap != cudaStreamCaptureStatusNone) return NEST_E_INVALID;   // no address yet: call once before capturing
        void *p = nullptr;
        if (int rc = nest::cuda_status(cudaGetSymbolAddress(&p, g_scratch), "cudaGetSymbolAddress")) return rc;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return NEST_OK;
}

}  // namespace

extern "C" int nest_solve_static(const nest_dims *dims, const void *records, int64_t *costs_out, void *plans_out,
                                 void *stream, const nest_options *opt) {
    if (!dims) return NEST_E_INVALID;
    if (opt && (opt->flags & NEST_KEEP_COSTS)) return NEST_E_INVALID;   // its tensor would be out of reach
    const size_t need = nest_workspace_size(dims, opt ? opt->chunk : 0);
    if (need == 0) return dims->B < 0 ? NEST_E_INVALID : NEST_E_LIMITS;
    if (need > size_t(NEST_STATIC_SCRATCH_BYTES)) return NEST_E_WORKSPACE;
    void *scratch = nullptr;
    if (int rc = scratch_address(stream, &scratch)) return rc;
    return nest_solve(dims, records, costs_out, plans_out, scratch, size_t(NEST_STATIC_SCRATCH_BYTES), stream, opt);
}
