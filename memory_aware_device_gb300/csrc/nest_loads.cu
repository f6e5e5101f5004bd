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
// GB300 mapping: one CTA per (instance, state i) copies the instance's derived tables
// (the prep block) into shared memory in one coalesced pass and takes the stages (i, j)
// for every j > i, a chunk of them at a time.  An item is one (stage, dense group): the
// strategies that share (t, cp) share the dense collective prices and those that also
// share e every expert one, so the thread of an item prices, per width, the dense
// gradient collectives once, the expert ones and the three amortised syncs once per e,
// and then evaluates each member's ZeRO stage and recompute choice with adds, selects
// and the memory test (unrolled when a group holds the whole (z, r) grid).  Each
// member's word is folded
// into a shared bucket[stage][m][pmax] with an atomic minimum on (tau << 16) | s (taken
// only when it improves the bucket); a suffix minimum over pmax gives the per-position
// loads.  The (stage, width, strategy) words themselves go to memory only when
// NEST_KEEP_COSTS asks for them.
#include <cuda_runtime.h>

#include "nest_stages.cuh"

namespace nest {

namespace {

constexpr int kThreads = 256;
constexpr int kBucketBytes = 48 * 1024;   // shared buckets per CTA, at most

__global__ void __launch_bounds__(kThreads) loads_kernel(PassArgs a, int pj_max) {
    extern __shared__ __align__(16) unsigned char smem[];   // prep block, buckets
    __shared__ uint32_t bmax_s;
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x, b = blockIdx.y;
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.ws + a.w.prep + int64_t(b) * a.w.prep_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int q = threadIdx.x; q < int(a.pl.bytes / 16); q += blockDim.x) dst[q] = src[q];
    }
    if (threadIdx.x == 0) bmax_s = 0;
    __syncthreads();
    const PrepHdr *ph = reinterpret_cast<const PrepHdr *>(smem);
    if (ph->status != NEST_SOLVED || i >= ph->L) return;   // uniform over the CTA
    const Geo &g = a.g;
    const int L = ph->L, K = ph->K, P = ph->P, ngd = ph->ngd;
    const int rowp = g.Pcap + 1;
    uint64_t *bucket = reinterpret_cast<uint64_t *>(smem + a.pl.bytes);
    const int npair = L - i;   // stages (i, j), j = i + 1 .. L
    int PJ = kThreads / ngd;
    PJ = PJ < 1 ? 1 : PJ > pj_max ? pj_max : PJ;
    uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride;
    const int64_t pos_stride = int64_t(g.NP) * g.Kpad;
    uint32_t tmax = 0;   // largest finite tau written, saturated at 2^31 - 1
    for (int c0 = 0; c0 < npair; c0 += PJ) {
        const int nj = PJ < npair - c0 ? PJ : npair - c0;
        for (int q = threadIdx.x; q < nj * g.Kmax * rowp; q += blockDim.x) bucket[q] = kInf;
        __syncthreads();
        for (int it = threadIdx.x; it < nj * ngd; it += blockDim.x) {
            const int jj = it / ngd, gd = it % ngd;
            const int j = i + 1 + c0 + jj;
            const int64_t pair = row_offset(i, L) + c0 + jj;
            uint64_t *bk = bucket + jj * g.Kmax * rowp;
            auto fold = [&](int m, int s, int64_t tau, int pm) {   // into bucket[m][pmax]
                if (pm == 0) return;   // also a strategy that does not apply (tau < 0)
                const uint64_t key = (uint64_t(tau) << 16) | uint64_t(s);
                uint64_t *slot = bk + m * rowp + pm;
                if (key < *slot) atomicMin(reinterpret_cast<unsigned long long *>(slot), key);
            };
            if (a.keep_costs) {
                uint64_t *cout = reinterpret_cast<uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                                 pair * g.Kmax * g.Spad;
                dense_group_words<true>(ph, smem, a.pl, g, i, j, gd, [&](int m, int s, int64_t tau, int pm) {
                    // the stage-cost word (tau << 8) | pmax, all ones where the strategy does not apply
                    cout[int64_t(m) * g.Spad + s] = tau < 0 ? kInf : (uint64_t(tau) << 8) | uint64_t(pm);
                    fold(m, s, tau, pm);
                });
            } else {
                dense_group_words<false>(ph, smem, a.pl, g, i, j, gd, fold);
            }
        }
        __syncthreads();
        // suffix minimum over pmax: position p takes the strategies with pmax >= p
        for (int r = threadIdx.x; r < nj * K; r += blockDim.x) {
            const int jj = r / K, m = r % K;
            const int64_t pr = row_offset(i, L) + c0 + jj;
            const uint64_t *bq = bucket + (jj * g.Kmax + m) * rowp;
            uint64_t cur = kInf;
            for (int p = P; p >= 1; p--) {
                cur = bq[p] < cur ? bq[p] : cur;
                out[int64_t(p - 1) * pos_stride + pr * g.Kpad + m] = cur;
                if (cur != kInf) {
                    const uint64_t tau = cur >> 16;
                    const uint32_t t32 = tau < 0x7FFFFFFFu ? uint32_t(tau) : 0x7FFFFFFFu;
                    tmax = t32 > tmax ? t32 : tmax;
                }
            }
        }
        __syncthreads();   // the buckets are reused
    }
    // one atomic per CTA: the sweeps keep 32-bit words when every value is small
    tmax = __reduce_max_sync(0xFFFFFFFFu, tmax);
    if ((threadIdx.x & 31) == 0 && tmax) atomicMax(&bmax_s, tmax);
    __syncthreads();
    if (threadIdx.x == 0 && bmax_s) atomicMax(&prep_hdr(a, b)->maxload32, bmax_s);
}

}  // namespace

int launch_loads(const PassArgs &a, void *stream) {
    // stages per chunk bounded by the shared buckets
    const int per_pair = a.g.Kmax * (a.g.Pcap + 1) * 8;
    int pj_max = kBucketBytes / per_pair;
    pj_max = pj_max < 1 ? 1 : pj_max > kThreads ? kThreads : pj_max;
    const size_t smem = size_t(a.pl.bytes) + size_t(pj_max) * per_pair;
    if (int rc = cuda_status(cudaFuncSetAttribute(loads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "loads smem attribute"))
        return rc;
    const dim3 grid(unsigned(a.g.Nmax), unsigned(a.n));
    return launch_kernel(loads_kernel, grid, dim3(kThreads), smem, stream, 1, "loads launch", a, pj_max);
}

}  // namespace nest
