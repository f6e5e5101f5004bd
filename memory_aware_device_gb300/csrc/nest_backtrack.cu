// Backtrack: the final batch-time loop and the stage reconstruction of Nest
// (Network- and Memory-Aware Device Placement) Appendix K Algorithm 1.
//
// t_batch = min over stage counts p of v(dp[0][Du][p]) * (M + p - 1) (ties to the
// smaller p), then the plan is read back by following the argument field of each
// DP cell: (j, m, c') gives the end of the stage, its width unit * 2^m and the
// candidate of its outgoing link; the stage's strategy is the argument of the
// per-position strategy minimum.  Lanes of a warp evaluate the stage counts in
// parallel and a shuffle reduction picks the best (t, p); lane 0 then walks the plan.
#include <cuda_runtime.h>

#include "nest_stages.cuh"

namespace nest {

namespace {

__global__ void __launch_bounds__(128) backtrack_kernel(PassArgs a) {
    __shared__ int walk[4][64];
    pdl_wait();
    pdl_trigger();
    const int b = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    if (b >= a.n) return;   // whole warps
    backtrack_warp(a, b, walk[threadIdx.x >> 5]);
}

}  // namespace

int launch_backtrack(const PassArgs &a, void *stream) {
    const int threads = 128;
    const int64_t total = int64_t(a.n) * 32;
    return launch_kernel(backtrack_kernel, dim3(unsigned((total + threads - 1) / threads)), dim3(threads), 0, stream, 1,
                         "backtrack launch", a);
}

}  // namespace nest
