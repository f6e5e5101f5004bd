// Joint search over variants of one problem: Nest (Network- and Memory-Aware Device
// Placement) §5.2.3 explores the microbatch size together with the placement; each
// variant is an instance of the batch and the search keeps, per group of
// consecutive variants, the one with the smallest t_batch (ties to the earlier one).
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

// One warp per group: lanes scan the group's variants, a shuffle reduction keeps
// the smallest (t_batch, index) among the solved ones (t_batch >= 0).
__global__ void __launch_bounds__(128) select_kernel(const int64_t *costs, int32_t groups, int32_t group,
                                                     int32_t *best) {
    pdl_wait();
    pdl_trigger();
    const int gi = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gi >= groups) return;   // whole warps
    long long bt = -1;
    int bq = -1;
    for (int q = lane; q < group; q += 32) {
        const long long t = costs[int64_t(gi) * group + q];
        if (t >= 0 && (bq < 0 || t < bt)) {
            bt = t;
            bq = q;
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        const long long ot = __shfl_xor_sync(0xffffffffu, bt, off);
        const int oq = __shfl_xor_sync(0xffffffffu, bq, off);
        if (oq >= 0 && (bq < 0 || ot < bt || (ot == bt && oq < bq))) {
            bt = ot;
            bq = oq;
        }
    }
    if (lane == 0) best[gi] = bq;
}

}  // namespace

}  // namespace nest

extern "C" int nest_select_best(const int64_t *costs, int32_t B, int32_t group, int32_t *best_out, void *stream) {
    if (B < 0 || group < 1 || B % group) return NEST_E_INVALID;
    if (B == 0) return NEST_OK;
    if (!costs || !best_out) return NEST_E_INVALID;
    const int32_t groups = B / group;
    const int threads = 128;
    const int64_t total = int64_t(groups) * 32;
    return nest::launch_kernel(nest::select_kernel, dim3(unsigned((total + threads - 1) / threads)), dim3(threads), 0,
                               stream, 1, "select launch", costs, groups, group, best_out);
}
