// Stage loads: the stage-cost builder and the per-position strategy reduction in
// one pass, loads[b][p-1][pair(i, j)][m] = min over the strategies s that fit
// position p of (tau << 16) | s.
//
// Nest (Network- and Memory-Aware Device Placement) §4 load(): the latency of a
// stage holding layers [i, j) on k = unit * 2^m devices under strategy s =
// (t, cp, e, z, r) is its compute scaled by the tensor/context degree, plus the
// tensor-, context- and expert-parallel collectives priced on the smallest tier
// that holds each group, plus ZeRO-3 weight gathers, all divided over the
// q = k / (t cp) data-parallel replicas, plus the gradient synchronisation
// amortised over the M microbatches of an iteration.  §3.3: the stage fits at
// pipeline position p while weights + gradients + optimizer states (each sharded
// by the ZeRO stage) + activations + (p - 1) stashed microbatches stay within the
// budget; pmax is the largest such p.  That is the 1F1B schedule; under GPipe the
// stash scales with B/d instead - every replica holds all of its ceil(M / q)
// microbatches at every position - so pmax is P or 0.  §4 Eq. 3 takes, for each
// new stage, the best latency over its strategies with memory-infeasible states
// pruned; the link terms of a transition do not depend on the strategy, so that
// minimum is taken once per (stage, width, position) - Appendix K Algorithm 1
// likewise evaluates a stage's load once before its inner loops.
//
// Arithmetic: every group size is a power of two, so each ceil-division by a group
// is a shift, and ceil((n - 1) phi V / n) = phi V - floor(phi V / n).  The
// remaining divisions (by a tier's bandwidth, by M and by R) use precomputed
// invariant divisors (Granlund & Montgomery, see nest_divide.cuh).  pmax comes
// from a float estimate corrected by exact integer comparisons.
//
// GB300 mapping: a CTA copies the instance's derived tables (the prep block) into
// shared memory in one coalesced pass and handles `ppc` stages (pairs); `spt`
// threads per stage run over its strategies.  A thread computes the width-free
// terms of one (stage, strategy) once and then its K width words, folding each into
// a shared bucket[pair][m][pmax] with an atomic minimum on (tau << 16) | s (taken
// only when it improves the bucket).  A suffix minimum over pmax gives the
// per-position loads.  The (stage, width, strategy) words themselves go to memory
// only when NEST_KEEP_COSTS asks for them.
#include <cuda_runtime.h>

#include "nest_stages.cuh"

namespace nest {

namespace {

constexpr int kThreads = 256;
constexpr int kBucketBytes = 64 * 1024;   // shared buckets per CTA, at most

__global__ void __launch_bounds__(kThreads) loads_kernel(PassArgs a, int spt, int ppc) {
    extern __shared__ __align__(16) unsigned char smem[];   // prep block, buckets, one word
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.ws + a.w.prep + int64_t(b) * a.w.prep_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int q = threadIdx.x; q < int(a.pl.bytes / 16); q += blockDim.x) dst[q] = src[q];
    }
    __syncthreads();
    if (reinterpret_cast<const PrepHdr *>(smem)->status != NEST_SOLVED) return;   // uniform over the CTA
    uint64_t *bucket = reinterpret_cast<uint64_t *>(smem + a.pl.bytes);
    uint32_t *bmax = reinterpret_cast<uint32_t *>(bucket + int64_t(ppc) * a.g.Kmax * (a.g.Pcap + 1));
    loads_slice(a, b, smem, int64_t(blockIdx.x) * ppc, ppc, spt, bucket, bmax);
}

}  // namespace

int launch_loads(const PassArgs &a, void *stream) {
    // spt threads per stage over its strategies, ppc stages per CTA (bounded by the
    // shared buckets)
    const int spt = a.g.Smax < kThreads ? a.g.Smax : kThreads;
    const int per_pair = a.g.Kmax * (a.g.Pcap + 1) * 8;
    int ppc = kThreads / spt;
    if (ppc * per_pair > kBucketBytes) ppc = kBucketBytes / per_pair > 0 ? kBucketBytes / per_pair : 1;
    const int threads = (ppc * spt + 31) / 32 * 32;
    const size_t smem = size_t(a.pl.bytes) + size_t(ppc) * per_pair + 16;
    if (int rc = cuda_status(cudaFuncSetAttribute(loads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "loads smem attribute"))
        return rc;
    const dim3 grid(unsigned((int64_t(a.g.NP) + ppc - 1) / ppc), unsigned(a.n));
    return launch_kernel(loads_kernel, grid, dim3(unsigned(threads)), smem, stream, 1, "loads launch", a, spt, ppc);
}

}  // namespace nest
