// Strategy reduction: loads[b][p-1][pair(i, j)][m] = min over strategies s whose
// memory fits position p of (tau << 16) | s.
//
// Nest (Network- and Memory-Aware Device Placement) §4 Eq. 3 takes, for each new
// stage, the best latency over its sub-graph strategies (the te superscript and
// load()), with memory-infeasible states pruned (§3.3: a stage at position p from
// the pipeline end holds p - 1 stashed microbatches).  Because the link terms of a
// transition do not depend on the strategy, the minimum over strategies can be
// taken once per (stage, width, position) - Appendix K Algorithm 1 likewise calls
// GETLOADOFSTAGE once per stage before its inner loops.
//
// One thread per row (pair, m) streams the row's S words with 16-byte loads and
// keeps, in its own shared-memory column, the smallest key per pmax value; a
// suffix minimum over pmax then gives every position at once.  The kernel reads
// the cost tensor exactly once (HBM-bound) and writes Pmax words per row.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) reduce_kernel(PassArgs a) {
    extern __shared__ uint64_t bucket[];   // [Pcap + 1][kThreads]
    const int b = blockIdx.y;
    const PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;
    const int L = ph->L, K = ph->K, S = ph->S, P = ph->P;
    const int64_t rows = int64_t(L) * (L + 1) / 2 * K;
    const int64_t row = int64_t(blockIdx.x) * kThreads + threadIdx.x;
    if (row >= rows) return;
    const int64_t pair = row / K;
    const int m = int(row % K);
    const uint64_t *src = reinterpret_cast<const uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                          (pair * a.g.Kmax + m) * a.g.Spad;
    uint64_t *col = bucket + threadIdx.x;
    for (int p = 1; p <= P; p++) col[p * kThreads] = kInf;
    const ulonglong2 *src2 = reinterpret_cast<const ulonglong2 *>(src);
    for (int s2 = 0; 2 * s2 < S; s2++) {
        const ulonglong2 v = __ldg(src2 + s2);
        const uint64_t w[2] = {v.x, v.y};
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int s = 2 * s2 + h;
            if (s < S && w[h] != kInf) {
                const int pm = int(w[h] & 0xFF);
                if (pm > 0) {
                    const uint64_t key = ((w[h] >> 8) << 16) | uint64_t(s);
                    if (key < col[pm * kThreads]) col[pm * kThreads] = key;
                }
            }
        }
    }
    uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride +
                    pair * a.g.Kpad + m;
    uint64_t cur = kInf;
    for (int p = P; p >= 1; p--) {
        const uint64_t v = col[p * kThreads];
        cur = v < cur ? v : cur;
        out[int64_t(p - 1) * a.g.NP * a.g.Kpad] = cur;
    }
}

}  // namespace

int launch_reduce(const PassArgs &a, void *stream) {
    const int64_t rows = int64_t(a.g.NP) * a.g.Kmax;
    const size_t smem = size_t(a.g.Pcap + 1) * kThreads * sizeof(uint64_t);
    if (int rc = cuda_status(cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "reduce smem attribute"))
        return rc;
    dim3 grid(unsigned((rows + kThreads - 1) / kThreads), unsigned(a.n));
    reduce_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(a);
    return cuda_status(cudaGetLastError(), "reduce launch");
}

}  // namespace nest
