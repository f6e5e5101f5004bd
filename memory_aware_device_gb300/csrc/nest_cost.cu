// Cost builder: fills cost[b][pair(i, j)][m][s] = (tau << 8) | pmax.
//
// Nest (Network- and Memory-Aware Device Placement) §4 load(): the latency of a
// stage holding layers [i, j) on k = unit * 2^m devices under strategy s =
// (t, cp, e, z, r) is its compute scaled by the tensor/context degree, plus the
// tensor-, context- and expert-parallel collectives priced on the smallest tier
// that holds each group, plus ZeRO-3 weight gathers, all divided over the
// q = k / (t cp) data-parallel replicas, plus the gradient synchronisation
// amortised over the M microbatches of an iteration.  §3.3: the stage fits at
// pipeline position p while weights + gradients + optimizer states (each
// sharded by the ZeRO stage) + activations + (p - 1) stashed microbatches stay
// within the budget; pmax is the largest such p.
//
// Arithmetic: every group size is a power of two, so each ceil-division by a
// group is a shift, and ceil((n - 1) phi V / n) = phi V - floor(phi V / n).  The
// remaining divisions (by a tier's bandwidth, by M and by R) use precomputed
// invariant divisors (Granlund & Montgomery, see nest_divide.cuh).  pmax comes
// from a float estimate corrected by exact integer comparisons.
//
// Layout: one thread per (pair, s) computes the width-independent terms once and
// then writes the K words of its (pair, *, s) column; consecutive threads hold
// consecutive s, so each of the K stores is coalesced over s.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

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

__global__ void __launch_bounds__(256) cost_kernel(PassArgs a) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;
    const int L = ph->L, S = ph->S, K = ph->K, lu = ph->lu;
    const int64_t total = int64_t(L) * (L + 1) / 2 * S;
    const int64_t gidx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gidx >= total) return;
    const int pair = int(gidx / S), s = int(gidx % S);
    // invert pair = row_offset(i) + (j - i - 1)
    int i = int((2.0f * L + 1.0f - sqrtf((2.0f * L + 1.0f) * (2.0f * L + 1.0f) - 8.0f * pair)) * 0.5f);
    if (i < 0) i = 0;
    if (i > L - 1) i = L - 1;
    while (i > 0 && row_offset(i, L) > pair) i--;
    while (i < L - 1 && row_offset(i + 1, L) <= pair) i++;
    const int j = i + 1 + int(pair - row_offset(i, L));

    uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                    int64_t(pair) * a.g.Kmax * a.g.Spad + s;
    const unsigned char *pb = reinterpret_cast<const unsigned char *>(ph);
    const uint32_t code = reinterpret_cast<const uint32_t *>(pb + a.pl.strat)[s];
    const int lt = code & 15, lcp = (code >> 4) & 15, le = (code >> 8) & 15;
    const int z = (code >> 12) & 3, r = (code >> 14) & 1;
    const int64_t *pfx = reinterpret_cast<const int64_t *>(pb + a.pl.pfx);
    const int64_t ld = a.g.Lmax + 1;
    const int64_t nM = pfx[kNm * ld + j] - pfx[kNm * ld + i];
    // valid for some width iff t cp e <= the widest stage, and e > 1 only over MoE layers
    const int lmin = lt + lcp + le - lu;  // smallest m that admits the strategy
    if (lmin > K - 1 || (le > 0 && nM == 0)) {
        for (int m = 0; m < K; m++) out[int64_t(m) * a.g.Spad] = kInf;
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
        const int64_t *ao = reinterpret_cast<const int64_t *>(pb + a.pl.ao);
        const int64_t *awst = reinterpret_cast<const int64_t *>(pb + a.pl.awst);
        const int lv = 31 - __clz(j - i);
        const int64_t m1 = awst[int64_t(lv) * a.g.Lmax + i], m2 = awst[int64_t(lv) * a.g.Lmax + j - (1 << lv)];
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
        out[int64_t(m) * a.g.Spad] = word;
    }
}

}  // namespace

int launch_cost(const PassArgs &a, void *stream) {
    const int64_t work = int64_t(a.g.NP) * a.g.Smax;
    const int threads = 256;
    dim3 grid(unsigned((work + threads - 1) / threads), unsigned(a.n));
    return launch_kernel(cost_kernel, grid, dim3(threads), 0, stream, 1, "cost launch", a);
}

}  // namespace nest
