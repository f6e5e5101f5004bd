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

#include "nest_internal.cuh"

namespace nest {

namespace {

constexpr int kThreads = 256;
constexpr int kBucketBytes = 64 * 1024;   // shared buckets per CTA, at most

__device__ __forceinline__ int64_t up_shift(int64_t x, int l) { return (x + (int64_t(1) << l) - 1) >> l; }

struct Net {
    const PrepHdr *ph;
    // Ring-model cost of cnt collectives moving V bytes in total over 2^ln devices on
    // tier tr; phi = 2 for AllReduce, 1 for AllGather / ReduceScatter / AllToAll.
    __device__ __forceinline__ int64_t coll(int64_t phi, int ln, int tr, int64_t V, int64_t cnt) const {
        if (ln == 0 || V == 0) return 0;
        const int64_t pv = phi * V;
        const int64_t per_device = pv - (pv >> ln);  // ceil(phi (n - 1) V / n)
        const int64_t steps = cnt * phi * ((int64_t(1) << ln) - 1) * ph->lat[tr];
        return steps + int64_t(divide_up(uint64_t(per_device) * 1000, uint64_t(ph->bw[tr]), ph->bwdiv[tr]));
    }
};

// The K width words (tau << 8) | pmax of stage [i, j) under strategy s, handed to
// emit(m, word); all ones where the strategy does not apply at that width.
template <typename Emit>
__device__ __forceinline__ void stage_words(const PrepHdr *ph, const unsigned char *pb, const PrepLayout &pl,
                                            const Geo &g, int i, int j, int s, Emit emit) {
    const int K = ph->K, lu = ph->lu;
    const uint32_t code = reinterpret_cast<const uint32_t *>(pb + pl.strat)[s];
    const int lt = code & 15, lcp = (code >> 4) & 15, le = (code >> 8) & 15;
    const int z = (code >> 12) & 3, r = (code >> 14) & 1;
    const int64_t *pfx = reinterpret_cast<const int64_t *>(pb + pl.pfx);
    const int64_t ld = g.Lmax + 1;
    const int64_t nM = pfx[kNm * ld + j] - pfx[kNm * ld + i];
    // valid for some width iff t cp e <= the widest stage, and e > 1 only over MoE layers
    const int lmin = lt + lcp + le - lu;  // smallest m that admits the strategy
    if (lmin > K - 1 || (le > 0 && nM == 0)) {
        for (int m = 0; m < K; m++) emit(m, kInf);
        return;
    }
    auto sum = [&](int q) { return pfx[q * ld + j] - pfx[q * ld + i]; };
    const int64_t Fl = sum(kFl), Pd = sum(kPd), Pe = sum(kPe), Ao = sum(kAo), Aw = sum(kAw), A2 = sum(kA2);
    const int64_t nL = j - i;
    const Net net{ph};

    // width-independent terms: groups inside one replica
    const int64_t comp = int64_t(divide_up(uint64_t(up_shift(Fl * (3 + r), lt + lcp)), uint64_t(ph->R), ph->Rdiv));
    const int64_t rep = comp + net.coll(2, lt, ph->tier_log[lt], 4 * up_shift(Ao, lcp), 4 * nL) +
                        net.coll(1, lcp, ph->tier_log[lt + lcp], 4 * up_shift(Ao, lt), 4 * nL) +
                        net.coll(1, le, ph->tier_log[lt + lcp + le], 4 * up_shift(A2, lt + lcp), 4 * nM);
    const int64_t Wd = up_shift(Pd, lt), We = up_shift(Pe, lt + le);
    int64_t act, stash;
    if (r) {
        const int64_t *ao = reinterpret_cast<const int64_t *>(pb + pl.ao);
        const int64_t *awst = reinterpret_cast<const int64_t *>(pb + pl.awst);
        const int lv = 31 - __clz(j - i);
        const int64_t m1 = awst[int64_t(lv) * g.Lmax + i], m2 = awst[int64_t(lv) * g.Lmax + j - (1 << lv)];
        act = up_shift(m1 > m2 ? m1 : m2, lt + lcp);
        stash = up_shift(i > 0 ? ao[i - 1] : ao[0], lt + lcp);
    } else {
        act = up_shift(Aw, lt + lcp);
        stash = act;
    }
    const int64_t opt = ph->opt, budget = ph->budget, M = ph->M;
    const int P = ph->P;
    const float inv_stash = stash > 0 ? 1.0f / float(stash) : 0.0f;
    const int64_t mult = z == 0 ? 1 : (z < 3 ? 2 : 1);
    const int64_t phi_s = z == 0 ? 2 : 1;
    for (int m = 0; m < K; m++) {
        uint64_t word = kInf;
        if (m >= lmin) {
            const int lq = lu + m - lt - lcp, lqe = lq - le;
            const int tk = ph->tier_log[lu + m];
            const int64_t z3 =
                z == 3 ? net.coll(1, lq, tk, 2 * Wd, 2 * nL) + net.coll(1, lqe, tk, 2 * We, 2 * nM) : 0;
            const int64_t sync = mult * (net.coll(phi_s, lq, tk, Wd, nL) + net.coll(phi_s, lqe, tk, We, nM));
            const int64_t tau = up_shift(rep + z3, lq) + int64_t(divide_up(uint64_t(sync), uint64_t(M), ph->Mdiv));
            if (tau < kCap) {
                const int64_t sh = up_shift(Wd, lq) + up_shift(We, lqe);
                const int64_t w = z == 3 ? sh : Wd + We;
                const int64_t gr = z >= 2 ? sh : Wd + We;
                const int64_t o = z >= 1 ? up_shift(opt * Wd, lq) + up_shift(opt * We, lqe) : opt * (Wd + We);
                const int64_t stat = w + gr + o + act;
                int pmax;
                if (stat > budget) {
                    pmax = 0;
                } else if (ph->schedule == 1) {
                    // GPipe: ceil(M / q) stashed microbatches; exact 128-bit product
                    const uint64_t inflight = uint64_t((M + (int64_t(1) << lq) - 1) >> lq);
                    const uint64_t lo = uint64_t(stash) * inflight, hi = __umul64hi(uint64_t(stash), inflight);
                    pmax = hi == 0 && lo <= uint64_t(budget - stat) ? P : 0;
                } else if (stash == 0) {
                    pmax = P;
                } else {
                    // largest p <= P with (p - 1) stash <= budget - stat
                    const int64_t rem = budget - stat;
                    int p = 1 + int(fminf(float(rem) * inv_stash, 64.0f));
                    p = p > P ? P : p;
                    while (p > 1 && int64_t(p - 1) * stash > rem) p--;
                    while (p < P && int64_t(p) * stash <= rem) p++;
                    pmax = p;
                }
                word = (uint64_t(tau) << 8) | uint64_t(pmax);
            }
        }
        emit(m, word);
    }
}

__global__ void __launch_bounds__(kThreads) loads_kernel(PassArgs a, int spt, int ppc) {
    extern __shared__ __align__(16) unsigned char smem[];   // prep block, then buckets
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const Geo &g = a.g;
    const PrepLayout &pl = a.pl;
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.ws + a.w.prep + int64_t(b) * a.w.prep_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int q = threadIdx.x; q < int(pl.bytes / 16); q += blockDim.x) dst[q] = src[q];
    }
    __syncthreads();
    const PrepHdr *ph = reinterpret_cast<const PrepHdr *>(smem);
    if (ph->status != NEST_SOLVED) return;   // uniform over the CTA
    const int L = ph->L, S = ph->S, K = ph->K, P = ph->P;
    const int64_t npairs = int64_t(L) * (L + 1) / 2;
    const int64_t pair0 = int64_t(blockIdx.x) * ppc;
    if (pair0 >= npairs) return;             // uniform over the CTA
    const int rowp = g.Pcap + 1;
    uint64_t *bucket = reinterpret_cast<uint64_t *>(smem + pl.bytes);   // [ppc][Kmax][Pcap + 1]
    for (int q = threadIdx.x; q < ppc * g.Kmax * rowp; q += blockDim.x) bucket[q] = kInf;
    __syncthreads();

    const int lp = threadIdx.x / spt, s0 = threadIdx.x % spt;
    const int64_t pair = pair0 + lp;
    if (lp < ppc && pair < npairs) {
        // invert pair = row_offset(i) + (j - i - 1)
        int i = int((2.0f * L + 1.0f - sqrtf((2.0f * L + 1.0f) * (2.0f * L + 1.0f) - 8.0f * float(pair))) * 0.5f);
        if (i < 0) i = 0;
        if (i > L - 1) i = L - 1;
        while (i > 0 && row_offset(i, L) > pair) i--;
        while (i < L - 1 && row_offset(i + 1, L) <= pair) i++;
        const int j = i + 1 + int(pair - row_offset(i, L));
        uint64_t *bk = bucket + lp * g.Kmax * rowp;
        uint64_t *cout = a.keep_costs ? reinterpret_cast<uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                                            pair * g.Kmax * g.Spad
                                      : nullptr;
        for (int s = s0; s < S; s += spt) {
            stage_words(ph, smem, pl, g, i, j, s, [&](int m, uint64_t w) {
                if (cout) cout[int64_t(m) * g.Spad + s] = w;
                const int pm = w == kInf ? 0 : int(w & 0xFF);
                if (pm == 0) return;
                const uint64_t key = ((w >> 8) << 16) | uint64_t(s);
                uint64_t *slot = bk + m * rowp + pm;
                if (key < *slot) atomicMin(reinterpret_cast<unsigned long long *>(slot), key);
            });
        }
    }
    __syncthreads();
    // suffix minimum over pmax: position p takes the strategies with pmax >= p
    uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride;
    const int64_t pos_stride = int64_t(g.NP) * g.Kpad;
    uint32_t tmax = 0;   // largest finite tau written, saturated at 2^31 - 1
    for (int r = threadIdx.x; r < ppc * K; r += blockDim.x) {
        const int q = r / K, m = r % K;
        const int64_t pr = pair0 + q;
        if (pr >= npairs) continue;
        const uint64_t *bq = bucket + (q * g.Kmax + m) * rowp;
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
    // one atomic per CTA: the sweep keeps 32-bit words when every value is small
    __shared__ uint32_t bmax;
    if (threadIdx.x == 0) bmax = 0;
    __syncthreads();
    tmax = __reduce_max_sync(0xFFFFFFFFu, tmax);
    if ((threadIdx.x & 31) == 0 && tmax) atomicMax(&bmax, tmax);
    __syncthreads();
    if (threadIdx.x == 0 && bmax) atomicMax(&prep_hdr(a, b)->maxload32, bmax);
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
    const size_t smem = size_t(a.pl.bytes) + size_t(ppc) * per_pair;
    if (int rc = cuda_status(cudaFuncSetAttribute(loads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "loads smem attribute"))
        return rc;
    const dim3 grid(unsigned((int64_t(a.g.NP) + ppc - 1) / ppc), unsigned(a.n));
    return launch_kernel(loads_kernel, grid, dim3(unsigned(threads)), smem, stream, 1, "loads launch", a, spt, ppc);
}

}  // namespace nest
