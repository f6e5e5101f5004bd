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
// Layout: one thread per (pair, s) computes the width-independent terms once and
// then writes the K words of its (pair, *, s) column; consecutive threads hold
// consecutive s, so each of the K stores is coalesced over s.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

struct Tiers {
    int T;
    const int64_t *G, *bw, *lat;
    __device__ __forceinline__ int of(int64_t n) const {
        int t = 0;
        while (t < T - 1 && G[t] < n) t++;
        return t;
    }
    // Ring-model cost of cnt collectives moving V bytes in total over n devices on
    // tier tr; phi = 2 for AllReduce, 1 for AllGather / ReduceScatter / AllToAll.
    __device__ __forceinline__ int64_t coll(int64_t phi, int64_t n, int tr, int64_t V, int64_t cnt) const {
        if (n == 1 || V == 0) return 0;
        const int64_t per_device = cdiv(phi * (n - 1) * V, n);
        return cnt * phi * (n - 1) * lat[tr] + cdiv(per_device * 1000, bw[tr]);
    }
};

__global__ void __launch_bounds__(256) cost_kernel(PassArgs a) {
    const int b = blockIdx.y;
    const PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;
    const int L = ph->L, S = ph->S, K = ph->K;
    const int64_t total = int64_t(L) * (L + 1) / 2 * S;
    const int64_t gidx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gidx >= total) return;
    const int pair = int(gidx / S), s = int(gidx % S);
    // invert pair = row_offset(i) + (j - i - 1)
    int i = int((2.0 * L + 1.0 - sqrt((2.0 * L + 1.0) * (2.0 * L + 1.0) - 8.0 * pair)) * 0.5);
    if (i < 0) i = 0;
    if (i > L - 1) i = L - 1;
    while (i > 0 && row_offset(i, L) > pair) i--;
    while (i < L - 1 && row_offset(i + 1, L) <= pair) i++;
    const int j = i + 1 + int(pair - row_offset(i, L));

    const unsigned char *pb = reinterpret_cast<const unsigned char *>(ph);
    const int64_t *pfx = reinterpret_cast<const int64_t *>(pb + a.pl.pfx);
    const int64_t ld = a.g.Lmax + 1;
    auto sum = [&](int q) { return pfx[q * ld + j] - pfx[q * ld + i]; };
    const int64_t Fl = sum(kFl), Pd = sum(kPd), Pe = sum(kPe), Ao = sum(kAo), Aw = sum(kAw),
                  A2 = sum(kA2), nM = sum(kNm), nL = j - i;
    const int64_t *ao = reinterpret_cast<const int64_t *>(pb + a.pl.ao);
    const int64_t ain = i > 0 ? ao[i - 1] : ao[0];
    const int64_t *awst = reinterpret_cast<const int64_t *>(pb + a.pl.awst);
    const int lv = 31 - __clz(j - i);
    const int64_t m1 = awst[int64_t(lv) * a.g.Lmax + i], m2 = awst[int64_t(lv) * a.g.Lmax + j - (1 << lv)];
    const int64_t AwMax = m1 > m2 ? m1 : m2;

    const uint32_t code = reinterpret_cast<const uint32_t *>(pb + a.pl.strat)[s];
    const int lt = code & 15, lcp = (code >> 4) & 15, le = (code >> 8) & 15;
    const int z = (code >> 12) & 3, r = (code >> 14) & 1;
    const int64_t t = int64_t(1) << lt, cp = int64_t(1) << lcp, e = int64_t(1) << le;
    const Tiers tr{ph->T, ph->G, ph->bw, ph->lat};

    // width-independent terms (groups inside one replica); skipped when no width
    // admits the strategy, which also keeps t cp R within 2^53
    const bool ep_ok = (e == 1 || nM > 0) && lt + lcp + le <= ph->lu + K - 1;
    int64_t rep = 0, Wd = 0, We = 0, act = 0, stash = 0;
    if (ep_ok) {
        const int64_t comp = cdiv(Fl * (3 + r), t * cp * ph->R);
        const int64_t tp = tr.coll(2, t, tr.of(t), 4 * cdiv(Ao, cp), 4 * nL);
        const int64_t cpc = tr.coll(1, cp, tr.of(t * cp), 4 * cdiv(Ao, t), 4 * nL);
        const int64_t ep = tr.coll(1, e, tr.of(t * cp * e), 4 * cdiv(A2, t * cp), 4 * nM);
        rep = comp + tp + cpc + ep;
        Wd = cdiv(Pd, t);
        We = cdiv(Pe, t * e);
        act = cdiv(r ? AwMax : Aw, t * cp);
        stash = cdiv(r ? ain : Aw, t * cp);
    }
    const int64_t opt = ph->opt, budget = ph->budget, P = ph->P, M = ph->M;
    uint64_t *out = reinterpret_cast<uint64_t *>(a.ws + a.w.cost) + int64_t(b) * a.w.cost_stride +
                    int64_t(pair) * a.g.Kmax * a.g.Spad + s;
    for (int m = 0; m < K; m++) {
        const int64_t k = int64_t(ph->unit) << m;
        uint64_t word = kInf;
        // valid iff t cp | k, e | q, and expert parallelism only over MoE layers
        if (ep_ok && lt + lcp + le <= ph->lu + m) {
            const int lq = ph->lu + m - lt - lcp;
            const int64_t q = int64_t(1) << lq, qe = int64_t(1) << (lq - le);
            const int tk = tr.of(k);
            int64_t z3 = 0, sd, se;
            if (z == 3) z3 = tr.coll(1, q, tk, 2 * Wd, 2 * nL) + tr.coll(1, qe, tk, 2 * We, 2 * nM);
            if (z == 0) {
                sd = tr.coll(2, q, tk, Wd, nL);
                se = tr.coll(2, qe, tk, We, nM);
            } else {
                const int64_t mult = z < 3 ? 2 : 1;
                sd = mult * tr.coll(1, q, tk, Wd, nL);
                se = mult * tr.coll(1, qe, tk, We, nM);
            }
            const int64_t tau = cdiv(rep + z3, q) + cdiv(sd + se, M);
            if (tau < kCap) {
                const int64_t sh = cdiv(Wd, q) + cdiv(We, qe);
                const int64_t w = z == 3 ? sh : Wd + We;
                const int64_t gr = z >= 2 ? sh : Wd + We;
                const int64_t o = z >= 1 ? cdiv(opt * Wd, q) + cdiv(opt * We, qe) : opt * (Wd + We);
                const int64_t stat = w + gr + o + act;
                int64_t pmax;
                if (stat > budget)
                    pmax = 0;
                else if (stash == 0)
                    pmax = P;
                else {
                    const int64_t f = 1 + (budget - stat) / stash;
                    pmax = f < P ? f : P;
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
    cost_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cuda_status(cudaGetLastError(), "cost launch");
}

}  // namespace nest
