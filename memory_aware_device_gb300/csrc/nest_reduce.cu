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
// A group of G lanes (G a power of two <= 32, chosen so that each lane reads a few
// words) reduces one row (pair, m) of S words: the lanes read the row with
// coalesced loads, each keeps in its own shared-memory column the smallest key per
// pmax value, takes a suffix minimum over pmax, and the group combines its lanes'
// columns per position.  The kernel reads the cost tensor once (HBM-bound) and
// writes Pmax words per row.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) reduce_kernel(PassArgs a, int lg) {
    extern __shared__ uint64_t bucket[];   // [Pcap + 1][kThreads], one column per lane
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;   // uniform over the block
    const int G = 1 << lg;
    const int L = ph->L, K = ph->K, S = ph->S, P = ph->P;
    const int64_t rows = int64_t(L) * (L + 1) / 2 * K;
    const int sub = threadIdx.x & (G - 1);
    const int64_t row = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> lg;
    const bool live = row < rows;
    const int64_t pair = live ? row / K : 0;
    const int m = live ? int(row % K) : 0;
    uint64_t *col = bucket + threadIdx.x;
    for (int p = 1; p <= P; p++) col[p * kThreads] = kInf;
    if (live) {
        const uint64_t *src = reinterpret_cast<const uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                              (pair * a.g.Kmax + m) * a.g.Spad;
        for (int s0 = sub; s0 < S; s0 += kUnroll * G) {
            uint64_t w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                const int s = s0 + u * G;
                w[u] = s < S ? __ldg(src + s) : kInf;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                if (w[u] == kInf) continue;
                const int pm = int(w[u] & 0xFF);
                if (pm == 0) continue;
                const uint64_t key = ((w[u] >> 8) << 16) | uint64_t(s0 + u * G);
                if (key < col[pm * kThreads]) col[pm * kThreads] = key;
            }
        }
        // suffix minimum: column entry p = best key among strategies with pmax >= p
        uint64_t cur = kInf;
        for (int p = P; p >= 1; p--) {
            const uint64_t v = col[p * kThreads];
            cur = v < cur ? v : cur;
            col[p * kThreads] = cur;
        }
    }
    __syncwarp();
    // lane `sub` of the group writes positions p = sub + 1, sub + 1 + G, ...
    uint32_t tmax = 0;   // largest finite tau written, saturated at 2^31 - 1
    if (live) {
        uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride +
                        pair * a.g.Kpad + m;
        const int base = threadIdx.x - sub;
        for (int p = sub + 1; p <= P; p += G) {
            uint64_t v = kInf;
            for (int q = 0; q < G; q++) {
                const uint64_t o = bucket[p * kThreads + base + q];
                v = o < v ? o : v;
            }
            out[int64_t(p - 1) * a.g.NP * a.g.Kpad] = v;
            if (v != kInf) {
                const uint64_t tau = v >> 16;
                const uint32_t t32 = tau < 0x7FFFFFFFu ? uint32_t(tau) : 0x7FFFFFFFu;
                tmax = t32 > tmax ? t32 : tmax;
            }
        }
    }
    // one atomic per block: the sweep uses 32-bit words when every value is small
    __shared__ uint32_t bmax;
    if (threadIdx.x == 0) bmax = 0;
    __syncthreads();
    tmax = __reduce_max_sync(0xFFFFFFFFu, tmax);
    if ((threadIdx.x & 31) == 0 && tmax) atomicMax(&bmax, tmax);
    __syncthreads();
    if (threadIdx.x == 0 && bmax) atomicMax(&ph->maxload32, bmax);
}

}  // namespace

int launch_reduce(const PassArgs &a, void *stream) {
    // lanes per row: about eight words per lane, at most a warp
    int lg = 0;
    while (lg < 5 && (8 << (lg + 1)) <= a.g.Smax) lg++;
    const int64_t rows = int64_t(a.g.NP) * a.g.Kmax;
    const int64_t rows_per_block = kThreads >> lg;
    const size_t smem = size_t(a.g.Pcap + 1) * kThreads * sizeof(uint64_t);
    if (int rc = cuda_status(cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "reduce smem attribute"))
        return rc;
    dim3 grid(unsigned((rows + rows_per_block - 1) / rows_per_block), unsigned(a.n));
    return launch_kernel(reduce_kernel, grid, dim3(kThreads), smem, stream, 1, "reduce launch", a, lg);
}

}  // namespace nest
