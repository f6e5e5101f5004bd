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

#include "nest_internal.cuh"

namespace nest {

namespace {

__device__ __forceinline__ bool pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }
__device__ __forceinline__ int ilog2(int64_t v) { return 63 - __clzll(v); }

__global__ void __launch_bounds__(256) prep_kernel(PassArgs a) {
    extern __shared__ __align__(16) unsigned char rec_s[];   // the instance's record
    pdl_wait();   // records and the workspace may still be in use by the previous kernel
    pdl_trigger();
    const int b = blockIdx.x;
    {   // one coalesced pass over the record; everything below reads shared memory
        const uint4 *src = reinterpret_cast<const uint4 *>(a.records + int64_t(b) * a.rl.record_bytes);
        uint4 *dst = reinterpret_cast<uint4 *>(rec_s);
        for (int q = threadIdx.x; q < int(a.rl.record_bytes / 16); q += blockDim.x) dst[q] = src[q];
    }
    __syncthreads();
    const unsigned char *rec = rec_s;
    const nest_record_header h = *reinterpret_cast<const nest_record_header *>(rec);
    PrepHdr *ph = prep_hdr(a, b);
    unsigned char *pb = reinterpret_cast<unsigned char *>(ph);
    const Geo &g = a.g;
    __shared__ int bad;
    if (threadIdx.x == 0) {
        int bd = 0;
        bd |= h.L < 1 || h.L > g.Lmax;
        bd |= !pow2(h.unit) || h.D < h.unit || h.D > 8192 || (h.unit > 0 && h.D % h.unit);
        bd |= h.unit > 0 && h.D / h.unit > g.Dumax;
        bd |= h.T < 1 || h.T > g.Tmax;
        bd |= h.C < 1 || h.C > g.Cmax;
        bd |= h.S < 1 || h.S > g.Smax;
        bd |= h.Pmax < 1 || h.Pmax > g.Pcap;
        bd |= h.M < h.Pmax || h.M > (int64_t(1) << 20);
        bd |= h.R < 1 || h.R > (int64_t(1) << 40);
        bd |= h.budget < 0 || h.budget > (int64_t(1) << 62);
        bd |= h.opt_factor < 0 || h.opt_factor > 16;
        bd |= h.schedule < 0 || h.schedule > 1;
        bad = bd;
    }
    __syncthreads();
    if (!bad) {
        const int64_t *G = reinterpret_cast<const int64_t *>(rec + a.rl.G);
        const int64_t *bw = reinterpret_cast<const int64_t *>(rec + a.rl.bw);
        const int64_t *lat = reinterpret_cast<const int64_t *>(rec + a.rl.lat);
        const int32_t *cand = reinterpret_cast<const int32_t *>(rec + a.rl.cand);
        const int16_t *st = reinterpret_cast<const int16_t *>(rec + a.rl.strat);
        int bd = 0;
        for (int l = threadIdx.x; l < h.L; l += blockDim.x) {
            const int64_t *arr[5] = {
                reinterpret_cast<const int64_t *>(rec + a.rl.pd), reinterpret_cast<const int64_t *>(rec + a.rl.pe),
                reinterpret_cast<const int64_t *>(rec + a.rl.ao), reinterpret_cast<const int64_t *>(rec + a.rl.aw),
                reinterpret_cast<const int64_t *>(rec + a.rl.a2a)};
            const int64_t f = reinterpret_cast<const int64_t *>(rec + a.rl.fl)[l];
            bd |= f < 0 || f > (int64_t(1) << 48);
            for (int q = 0; q < 5; q++) bd |= arr[q][l] < 0 || arr[q][l] > (int64_t(1) << 38);
            bd |= rec[a.rl.moe + l] > 1;
        }
        for (int t = threadIdx.x; t < h.T; t += blockDim.x) {
            bd |= !pow2(G[t]) || (t > 0 && G[t] <= G[t - 1]);
            bd |= bw[t] < 1000 || bw[t] > (int64_t(1) << 40);
            bd |= lat[t] < 0 || lat[t] > (int64_t(1) << 24);
        }
        if (threadIdx.x == 0) bd |= G[h.T - 1] < h.D;
        for (int c = threadIdx.x; c < h.C; c += blockDim.x) {
            bd |= cand[c] < 0 || cand[c] >= h.T || (c > 0 && cand[c] <= cand[c - 1]);
        }
        for (int s = threadIdx.x; s < h.S; s += blockDim.x) {
            const int16_t *x = st + 8 * s;
            for (int f = 0; f < 3; f++) bd |= !pow2(x[f]) || x[f] > 8192;
            bd |= x[3] < 0 || x[3] > 3 || x[4] < 0 || x[4] > 1;
        }
        bd = __syncthreads_or(bd);
        if (threadIdx.x == 0) bad = bd;
        __syncthreads();
    }
    if (bad) {
        if (threadIdx.x == 0) ph->status = NEST_BAD_INPUT;
        return;
    }

    const int L = h.L;
    const int64_t Du = h.D / h.unit;
    if (threadIdx.x == 0) {
        ph->L = L;
        ph->D = h.D;
        ph->unit = h.unit;
        ph->lu = ilog2(h.unit);
        ph->Du = int32_t(Du);
        ph->K = ilog2(Du) + 1;
        ph->T = h.T;
        ph->C = h.C;
        ph->S = h.S;
        ph->P = h.Pmax;
        ph->R = h.R;
        ph->M = h.M;
        ph->budget = h.budget;
        ph->opt = h.opt_factor;
        ph->schedule = h.schedule;
    }
    const int64_t *G = reinterpret_cast<const int64_t *>(rec + a.rl.G);
    const int64_t *bw = reinterpret_cast<const int64_t *>(rec + a.rl.bw);
    const int64_t *lat = reinterpret_cast<const int64_t *>(rec + a.rl.lat);
    const int32_t *cand = reinterpret_cast<const int32_t *>(rec + a.rl.cand);
    for (int t = threadIdx.x; t < 8; t += blockDim.x) {
        ph->G[t] = t < h.T ? G[t] : 0;
        ph->bw[t] = t < h.T ? bw[t] : 1;
        ph->lat[t] = t < h.T ? lat[t] : 0;
        ph->bwdiv[t] = make_divisor(uint64_t(t < h.T ? bw[t] : 1));
    }
    if (threadIdx.x == 8) ph->Mdiv = make_divisor(uint64_t(h.M));
    if (threadIdx.x == 9) ph->Rdiv = make_divisor(uint64_t(h.R));
    for (int x = threadIdx.x; x < 16; x += blockDim.x) {
        int t = 0;
        while (t < h.T - 1 && G[t] < (int64_t(1) << x)) t++;
        ph->tier_log[x] = int8_t(t);
    }
    for (int c = threadIdx.x; c < 16; c += blockDim.x) {
        int ml = -1;
        if (c < h.C) {
            const int64_t cap = G[cand[c]];
            for (int m = 0; m < 16; m++)
                if (2 * (int64_t(h.unit) << m) <= cap) ml = m;
        }
        ph->cand[c] = c < h.C ? cand[c] : 0;
        ph->mlim[c] = ml;
    }

    // prefix sums and the sparse table, built in shared memory (L <= 255): the layer
    // arrays are read once with coalesced loads, each array is scanned by one warp,
    // and the results are written back with coalesced stores
    __shared__ int64_t sv[kNumPfx][256];   // layer values, scanned in place
    __shared__ int64_t sst[kLogL][256];    // sparse table of max(aw)
    int64_t *pfx = reinterpret_cast<int64_t *>(pb + a.pl.pfx);
    int64_t *ao = reinterpret_cast<int64_t *>(pb + a.pl.ao);
    int64_t *awst = reinterpret_cast<int64_t *>(pb + a.pl.awst);
    {
        const int64_t off[6] = {a.rl.fl, a.rl.pd, a.rl.pe, a.rl.ao, a.rl.aw, a.rl.a2a};
        for (int e = threadIdx.x; e < kNumPfx * L; e += blockDim.x) {
            const int q = e / L, l = e % L;
            const int64_t v = q == kNm ? int64_t(rec[a.rl.moe + l]) : reinterpret_cast<const int64_t *>(rec + off[q])[l];
            sv[q][l] = v;
            if (q == kAw) sst[0][l] = v;
            if (q == kAo) ao[l] = v;
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kNumPfx) {
        int64_t carry = 0;
        for (int base = 0; base < L; base += 32) {
            int64_t x = base + lane < L ? sv[warp][base + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            x += carry;
            if (base + lane < L) sv[warp][base + lane] = x;
            carry = __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
    for (int lv = 1; lv < kLogL; lv++) {
        const int span = 1 << (lv - 1);
        for (int l = threadIdx.x; l < L; l += blockDim.x) {
            const int64_t x = sst[lv - 1][l];
            const int64_t y = l + span < L ? sst[lv - 1][l + span] : x;
            sst[lv][l] = x > y ? x : y;
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < kNumPfx * (L + 1); e += blockDim.x) {
        const int q = e / (L + 1), l = e % (L + 1);
        pfx[int64_t(q) * (g.Lmax + 1) + l] = l == 0 ? 0 : sv[q][l - 1];
    }
    for (int e = threadIdx.x; e < kLogL * L; e += blockDim.x) {
        const int lv = e / L, l = e % L;
        awst[int64_t(lv) * g.Lmax + l] = sst[lv][l];
    }
    const int64_t *ao_in = reinterpret_cast<const int64_t *>(rec + a.rl.ao);
    int64_t *X = reinterpret_cast<int64_t *>(pb + a.pl.X);
    __shared__ uint32_t xmax;
    if (threadIdx.x == 0) xmax = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < (L + 1) * h.C; e += blockDim.x) {
        const int bnd = e / h.C, c = e % h.C;
        int64_t v = 0;
        if (bnd > 0 && bnd < L) {
            const int tr = cand[c];
            v = lat[tr] + cdiv(ao_in[bnd - 1] * 1000, bw[tr]);
        }
        X[int64_t(bnd) * g.Cmax + c] = v;
        atomicMax(&xmax, v < 0x7FFFFFFF ? uint32_t(v) : 0x7FFFFFFFu);
    }
    uint32_t *sp = reinterpret_cast<uint32_t *>(pb + a.pl.strat);
    const int16_t *st = reinterpret_cast<const int16_t *>(rec + a.rl.strat);
    for (int s = threadIdx.x; s < h.S; s += blockDim.x) {
        const int16_t *x = st + 8 * s;
        sp[s] = uint32_t(ilog2(x[0])) | uint32_t(ilog2(x[1])) << 4 | uint32_t(ilog2(x[2])) << 8 |
                uint32_t(x[3]) << 12 | uint32_t(x[4]) << 14;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ph->maxX32 = xmax;
        ph->maxload32 = 0;   // raised by the strategy reduction
        ph->status = NEST_SOLVED;
    }
}

}  // namespace

int launch_prep(const PassArgs &a, void *stream) {
    const size_t smem = size_t(a.rl.record_bytes);
    if (int rc = cuda_status(cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "prep smem attribute"))
        return rc;
    return launch_kernel(prep_kernel, dim3(unsigned(a.n)), dim3(256), smem, stream, 1, "prep launch", a);
}

}  // namespace nest
