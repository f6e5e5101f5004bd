// Prep kernel: validates each instance and derives the per-instance tables the
// cost builder and the DP sweep read.
//
// Nest (Network- and Memory-Aware Device Placement) §3.2: the solver receives the
// operator chain annotated with per-layer compute, parameter and activation sizes
// plus the tiered network description (Appendix B).  This kernel turns those
// inputs into prefix sums over layers (stage sums in O(1)), a sparse table for
// the largest working activation of a stage, the link cost of every layer
// boundary over every candidate tier (the forward / backward traffic terms of
// §4 load()), and packed strategy codes.  One CTA per instance.
#include <cuda_runtime.h>

#include "nest_stages.cuh"

namespace nest {

namespace {

__global__ void __launch_bounds__(256) prep_kernel(PassArgs a) {
    extern __shared__ __align__(128) unsigned char scr[];
    pdl_wait();   // records and the workspace may still be in use by the previous kernel
    pdl_trigger();
    prep_instance(a, blockIdx.x, scr);
}

}  // namespace

int launch_prep(const PassArgs &a, void *stream) {
    const size_t smem = size_t(prep_scratch(a.g, a.rl).bytes);
    if (int rc = cuda_status(cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "prep smem attribute"))
        return rc;
    return launch_kernel(prep_kernel, dim3(unsigned(a.n)), dim3(256), smem, stream, 1, "prep launch", a);
}

}  // namespace nest
