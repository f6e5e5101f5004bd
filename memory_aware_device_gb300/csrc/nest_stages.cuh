// Device bodies shared by the pass kernels: the prep of one instance, the stage
// loads of a range of its stages, and its backtrack.  The standalone kernels
// (nest_prep.cu, nest_loads.cu, nest_backtrack.cu) run them one after the other;
// the fused resident sweep (nest_sweep.cu) runs all of them inside one launch.
//
// Nest (Network- and Memory-Aware Device Placement): §3.2 (per-layer metadata), §3.3
// (memory model, stash by schedule), §4 load() and Eq. 3 (stage latency, link terms,
// strategy minimum per stage), Appendix K Algorithm 1 (final batch-time loop and
// stage reconstruction); see the three kernel files for the details of each step.
#pragma once

#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

// Shared scratch of prep_instance: flags and counters, the record, the layer values,
// the sparse table and the up-set lists of a graph instance (byte offsets).
struct PrepScratch {
    int64_t flags, rec, sv, sst, gen, lev, sain, sdiv, bytes;
};

__host__ __device__ inline PrepScratch prep_scratch(const Geo &g, const nest_layout &rl) {
    PrepScratch s;
    s.flags = 0;
    s.rec = 128;
    s.sv = s.rec + align_up(rl.record_bytes, 128);
    s.sst = s.sv + align_up(8 * int64_t(kNumPfx) * g.Lmax, 128);
    s.gen = s.sst + align_up(8 * int64_t(kLogL) * g.Lmax, 128);
    s.lev = s.gen + 8 * kMaxStates;
    s.sain = s.lev + 4 * 72;                          // bytes entering each state
    s.sdiv = s.sain + 8 * kMaxStates;                 // the tier divisors
    s.bytes = s.sdiv + int64_t(sizeof(Divisor)) * 8;
    return s;
}

__device__ __forceinline__ bool pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }
__device__ __forceinline__ int ilog2(int64_t v) { return 63 - __clzll(v); }
__device__ __forceinline__ uint64_t low_bits(int n) { return n >= 64 ? ~uint64_t(0) : (uint64_t(1) << n) - 1; }

// The prep of instance b (validation, prefix sums, sparse table, link table,
// strategy codes, invariant divisors) into its prep block in the workspace, using
// `scr` (prep_scratch bytes of shared memory).  Every thread of the block calls it.
static __device__ __noinline__ void prep_instance(const PassArgs &a, int b, unsigned char *scr) {
    const PrepScratch ps = prep_scratch(a.g, a.rl);
    int &bad = *reinterpret_cast<int *>(scr + ps.flags);
    uint32_t &xmax = *reinterpret_cast<uint32_t *>(scr + ps.flags + 4);
    unsigned char *rec_s = scr + ps.rec;
    int64_t *sv = reinterpret_cast<int64_t *>(scr + ps.sv);     // [kNumPfx][Lmax], scanned in place
    int64_t *sst = reinterpret_cast<int64_t *>(scr + ps.sst);   // [kLogL][Lmax], sparse table of max(aw)
    const int LM = a.g.Lmax;
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
        bd |= h.graph < 0 || h.graph > 1;
        bd |= h.graph == 1 && (h.L > 63 || g.Vmax < 1);
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
            if (h.graph)   // edges go forward, to layers of the instance
                bd |= (reinterpret_cast<const uint64_t *>(rec + a.rl.succ)[l] & ~(low_bits(h.L) & ~low_bits(l + 1))) != 0;
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
        ph->layers = L;
        ph->graph = h.graph;
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
    }
    // the invariant divisors (the tiers' bandwidths, M and R), one per warp's lane 0 so
    // that they are computed side by side; the tier divisors are kept in shared memory
    // for the link table too
    Divisor *sdiv = reinterpret_cast<Divisor *>(scr + ps.sdiv);
    if ((threadIdx.x & 31) == 0)
        for (int k = int(threadIdx.x >> 5); k < 10; k += int(blockDim.x >> 5)) {
            // k < T: tier k; T: M; T + 1: R; beyond: the unused tiers (divisor 1)
            if (k < h.T) {
                sdiv[k] = make_divisor(uint64_t(bw[k]));
                ph->bwdiv[k] = sdiv[k];
            } else if (k == h.T) {
                ph->Mdiv = make_divisor(uint64_t(h.M));
            } else if (k == h.T + 1) {
                ph->Rdiv = make_divisor(uint64_t(h.R));
            } else {
                const int t = k - 2;   // h.T <= t < 8
                ph->bwdiv[t] = make_divisor(1);
            }
        }
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

    // prefix sums and the sparse table, built in shared memory: the layer arrays are
    // read once with coalesced loads, each array is scanned by one warp, and the
    // results are written back with coalesced stores
    int64_t *pfx = reinterpret_cast<int64_t *>(pb + a.pl.pfx);
    int64_t *awst = reinterpret_cast<int64_t *>(pb + a.pl.awst);
    {
        const int64_t off[6] = {a.rl.fl, a.rl.pd, a.rl.pe, a.rl.ao, a.rl.aw, a.rl.a2a};
        for (int e = threadIdx.x; e < kNumPfx * L; e += blockDim.x) {
            const int q = e / L, l = e % L;
            const int64_t v = q == kNm ? int64_t(rec[a.rl.moe + l]) : reinterpret_cast<const int64_t *>(rec + off[q])[l];
            sv[q * LM + l] = v;
            if (q == kAw) sst[l] = v;
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int q = warp; q < kNumPfx; q += int(blockDim.x >> 5)) {
        int64_t carry = 0;
        for (int base = 0; base < L; base += 32) {
            int64_t x = base + lane < L ? sv[q * LM + base + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            x += carry;
            if (base + lane < L) sv[q * LM + base + lane] = x;
            carry = __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
    for (int lv = 1; lv < kLogL; lv++) {
        const int span = 1 << (lv - 1);
        for (int l = threadIdx.x; l < L; l += blockDim.x) {
            const int64_t x = sst[(lv - 1) * LM + l];
            const int64_t y = l + span < L ? sst[(lv - 1) * LM + l + span] : x;
            sst[lv * LM + l] = x > y ? x : y;
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < kNumPfx * (L + 1); e += blockDim.x) {
        const int q = e / (L + 1), l = e % (L + 1);
        pfx[int64_t(q) * (g.Lmax + 1) + l] = l == 0 ? 0 : sv[q * LM + l - 1];
    }
    for (int e = threadIdx.x; e < kLogL * L; e += blockDim.x) {
        const int lv = e / L, l = e % L;
        awst[int64_t(lv) * g.Lmax + l] = sst[lv * LM + l];
    }
    // the DP states: suffixes [b, L) of a chain, the up-sets of a graph; per state its
    // layer mask, the bytes entering it and the link cost into it per candidate
    const int64_t *ao_in = reinterpret_cast<const int64_t *>(rec + a.rl.ao);
    int64_t *ain = reinterpret_cast<int64_t *>(pb + a.pl.ain);
    int64_t *sain = reinterpret_cast<int64_t *>(scr + ps.sain);   // the same, in shared memory
    uint64_t *um = reinterpret_cast<uint64_t *>(pb + a.pl.umask);
    int E = L;   // the last state, the empty set
    if (!h.graph) {
        for (int q = threadIdx.x; q <= L; q += blockDim.x) {
            sain[q] = ain[q] = q > 0 ? ao_in[q - 1] : ao_in[0];
            um[q] = L <= 64 ? low_bits(L) & ~low_bits(q) : 0;
        }
    } else {
        // Up-sets grown by size: the children of D are D + {l} for each layer l below
        // the lowest layer of D whose successors all lie in D.  The lowest layer of an
        // up-set has no predecessor inside it (the numbering is topological), so
        // every up-set has exactly one parent and each is generated once.
        const uint64_t *succ = reinterpret_cast<const uint64_t *>(rec + a.rl.succ);
        uint64_t *gen = reinterpret_cast<uint64_t *>(scr + ps.gen);
        int *lev = reinterpret_cast<int *>(scr + ps.lev);   // level k is gen[lev[k] .. lev[k + 1])
        int &ngen = *reinterpret_cast<int *>(scr + ps.flags + 8);
        const int cap = g.Vmax + 1;   // <= kMaxStates
        if (threadIdx.x == 0) {
            gen[0] = 0;
            lev[0] = 0;
            lev[1] = 1;
            ngen = 1;
        }
        __syncthreads();
        for (int k = 0; k <= L; k++) {
            const int lo = lev[k], hi = lev[k + 1];
            if (lo == hi) break;   // uniform: shared values after a barrier
            for (int q = lo + int(threadIdx.x); q < hi; q += blockDim.x) {
                const uint64_t D = gen[q];
                const int top = D ? __ffsll((long long)D) - 1 : L;
                for (int l = 0; l < top; l++)
                    if ((succ[l] & ~D) == 0) {
                        const int at = atomicAdd(&ngen, 1);
                        if (at < cap) gen[at] = D | (uint64_t(1) << l);
                    }
            }
            __syncthreads();
            if (threadIdx.x == 0) lev[k + 2] = ngen < cap ? ngen : cap;
            __syncthreads();
        }
        const int n = ngen;
        if (n > cap) {   // more up-sets than the batch was sized for
            if (threadIdx.x == 0) ph->status = NEST_BAD_INPUT;
            return;
        }
        // state order: size descending, then mask ascending
        for (int e = threadIdx.x; e < n; e += blockDim.x) {
            int k = 0;
            while (lev[k + 1] <= e) k++;
            const uint64_t D = gen[e];
            int r = 0;
            for (int q = lev[k]; q < lev[k + 1]; q++) r += gen[q] < D;
            um[n - lev[k + 1] + r] = D;
        }
        __syncthreads();
        uint64_t fed = 0;   // layers with a predecessor
        for (int l = 0; l < L; l++) fed |= succ[l];
        const uint64_t full = low_bits(L);
        for (int q = threadIdx.x; q < n; q += blockDim.x) {
            const uint64_t D = um[q];
            int64_t v = 0;
            for (int l = 0; l < L; l++) {
                const uint64_t bit = uint64_t(1) << l;
                if (D == full ? !(fed & bit) : (!(D & bit) && (succ[l] & D))) v += ao_in[l];
            }
            sain[q] = ain[q] = v;
        }
        E = n - 1;
    }
    int64_t *X = reinterpret_cast<int64_t *>(pb + a.pl.X);
    if (threadIdx.x == 0) xmax = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < (E + 1) * h.C; e += blockDim.x) {
        const int q = e / h.C, c = e % h.C;
        int64_t v = 0;
        if (q > 0 && q < E) {
            const int tr = cand[c];
            v = lat[tr] + int64_t(divide_up(uint64_t(sain[q]) * 1000, uint64_t(bw[tr]), sdiv[tr]));
        }
        X[int64_t(q) * g.Cmax + c] = v;
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
    // the strategies sorted by (t, cp, e, z, r, s), and the groups of equal (t, cp, e): the
    // stage-loads pass prices the collectives of a group once per width and then each
    // member's ZeRO stage and recompute choice
    {
        uint32_t *ss = reinterpret_cast<uint32_t *>(pb + a.pl.ssort);
        uint32_t *sg = reinterpret_cast<uint32_t *>(pb + a.pl.sgrp);
        auto key = [&](int s) {
            const uint32_t c = sp[s];
            return uint64_t((c & 0xFFF) << 3 | (c >> 12 & 3) << 1 | (c >> 14 & 1)) << 12 | uint64_t(s);
        };
        for (int s = threadIdx.x; s < h.S; s += blockDim.x) {
            const uint64_t ks = key(s);
            int rank = 0;
            for (int t = 0; t < h.S; t++) rank += key(t) < ks;
            ss[rank] = sp[s] | uint32_t(s) << 16;
        }
        __syncthreads();
        uint32_t *sd = reinterpret_cast<uint32_t *>(pb + a.pl.sgd);
        if (threadIdx.x == 0) {
            int n = 0, nd = 0;
            for (int q = 0; q < h.S; q++) {
                if (q == 0 || (ss[q] & 0xFF) != (ss[q - 1] & 0xFF)) sd[nd++] = uint32_t(n);   // new (t, cp)
                if (q == 0 || (ss[q] & 0xFFF) != (ss[q - 1] & 0xFFF)) sg[n++] = uint32_t(q);  // new (t, cp, e)
            }
            sg[n] = uint32_t(h.S);
            sd[nd] = uint32_t(n);
            ph->ngrp = n;
            ph->ngd = nd;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ph->L = E;
        ph->maxX32 = xmax;
        ph->maxload32 = 0;   // raised by the strategy reduction
        ph->lay_sat = 0;
        ph->status = NEST_SOLVED;
    }
}


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
    // coll(1, ...) and coll(2, ...) of the same group, tier and bytes with one division:
    // the phi = 2 bytes per device are 2 x1 - b with x1 = V - floor(V / n) and
    // b = bit (ln - 1) of V, so with x1 * 1000 = q bw + r their ceiling over bw is
    // 2q + ceil(y / bw), y = 2r - 1000 b, and -bw <= -1000 <= y < 2 bw (bw >= 1000).
    __device__ __forceinline__ void coll12(int ln, int tr, int64_t V, int64_t cnt, int64_t &c1, int64_t &c2) const {
        if (ln == 0 || V == 0) {
            c1 = c2 = 0;
            return;
        }
        const int64_t x1 = V - (V >> ln);
        const int64_t steps = cnt * ((int64_t(1) << ln) - 1) * ph->lat[tr];
        const int64_t bw = ph->bw[tr];
        const int64_t q = int64_t(divide(uint64_t(x1) * 1000, ph->bwdiv[tr]));
        const int64_t r = x1 * 1000 - q * bw;
        const int64_t y = 2 * r - 1000 * ((V >> (ln - 1)) & 1);
        c1 = steps + q + (r > 0);
        c2 = 2 * steps + 2 * q + (y > bw ? 2 : y > 0 ? 1 : y > -bw ? 0 : -1);
    }
};

// Largest aw over layers [x, y), x < y, from the sparse table.
__device__ __forceinline__ int64_t aw_max(const int64_t *awst, const Geo &g, int x, int y) {
    const int lv = 31 - __clz(y - x);
    const int64_t m1 = awst[int64_t(lv) * g.Lmax + x], m2 = awst[int64_t(lv) * g.Lmax + y - (1 << lv)];
    return m1 > m2 ? m1 : m2;
}

// Per-layer metadata summed over a stage (§3.2), with its largest working activation.
struct StageSums {
    int64_t v[kNumPfx];   // kFl .. kNm
    int64_t nL, awmax;
};

// The sums of the layers in `S`: one prefix-sum difference and one sparse-table
// query per run of consecutive layers.  S < 2^63.
__device__ __forceinline__ void mask_sums(const int64_t *pfx, const int64_t *awst, const Geo &g, uint64_t S,
                                          StageSums &u) {
    const int64_t ld = g.Lmax + 1;
    for (int q = 0; q < kNumPfx; q++) u.v[q] = 0;
    u.nL = __popcll(S);
    u.awmax = 0;
    while (S) {
        const int x = __ffsll((long long)S) - 1;
        const int run = __ffsll((long long)~(S >> x)) - 1;   // bit 63 of S is clear, so run <= 63
        const int y = x + run;
        for (int q = 0; q < kNumPfx; q++) u.v[q] += pfx[q * ld + y] - pfx[q * ld + x];
        const int64_t mx = aw_max(awst, g, x, y);
        u.awmax = mx > u.awmax ? mx : u.awmax;
        S &= ~(low_bits(run) << x);
    }
}

// The stage sums of the stage from state i to state j: false when it is no stage (for a
// graph instance, state j not inside state i).
__device__ __forceinline__ bool pair_sums(const PrepHdr *ph, const unsigned char *pb, const PrepLayout &pl,
                                          const Geo &g, int i, int j, StageSums &u) {
    const int64_t *pfx = reinterpret_cast<const int64_t *>(pb + pl.pfx);
    const int64_t *awst = reinterpret_cast<const int64_t *>(pb + pl.awst);
    if (ph->graph) {
        const uint64_t *um = reinterpret_cast<const uint64_t *>(pb + pl.umask);
        const uint64_t Di = um[i], Dj = um[j];
        if (Dj & ~Di) return false;
        mask_sums(pfx, awst, g, Di & ~Dj, u);
        return true;
    }
    const int64_t ld = g.Lmax + 1;
    for (int q = 0; q < kNumPfx; q++) u.v[q] = pfx[q * ld + j] - pfx[q * ld + i];
    u.nL = j - i;
    u.awmax = aw_max(awst, g, i, j);
    return true;
}

// pmax of one strategy (§3.3): the largest position p <= P whose stash still fits,
// 1F1B (p - 1 stashed microbatches) or GPipe (all ceil(M / q) of a replica's).
// rem = budget - static >= 0; full = (P - 1) * stash, inv ~ 1 / stash.
__device__ __forceinline__ int fit_positions(const PrepHdr *ph, bool gpipe, int P, int64_t rem, int64_t st,
                                             int64_t full, float inv, int lq) {
    if (gpipe) {
        // GPipe: ceil(M / q) stashed microbatches; exact 128-bit product
        const uint64_t inflight = uint64_t((ph->M + (int64_t(1) << lq) - 1) >> lq);
        const uint64_t lo = uint64_t(st) * inflight, hi = __umul64hi(uint64_t(st), inflight);
        return hi == 0 && lo <= uint64_t(rem) ? P : 0;
    }
    if (rem >= full) return P;   // also st == 0
    // (P - 1) st > rem: the quotient is below 31; a float estimate, corrected exactly
    int p = 1 + int(float(rem) * inv);
    p = p > P ? P : p < 1 ? 1 : p;
    if (int64_t(p - 1) * st > rem) p--;
    else if (p < P && int64_t(p) * st <= rem) p++;
    return p;
}

// The stage time tau and the fitting positions pmax of stage (i, j) for every strategy
// of dense group gd (equal t, cp), handed to emit(m, s, tau, pmax) for every width m;
// tau = -1 where a strategy does not apply to a width or reaches the cap.  A dense group is a run of strategy groups (equal
// t, cp, e) whose members differ in the ZeRO stage z and recompute r.  Per width the
// collectives are priced once: the dense ones once per dense group, the expert ones
// once per strategy group.  With S1 = coll(1, q) + coll(1, q / e) and
// S2 = coll(2, q) + coll(2, q / e) over the dense and expert gradient bytes, the
// gradient sync is S2 for z = 0 (AllReduce), 2 S1 for z = 1, 2 (ReduceScatter +
// AllGather) and S1 for z = 3 (ReduceScatter); the ZeRO-3 weight gathers (two
// AllGathers of the shards per layer, count 2 nL and volume 2 W) cost exactly S2: the
// same latency steps (cnt phi) and the same bytes per device (phi V).
template <bool kAll, typename Emit>
__device__ __forceinline__ void dense_group_words(const PrepHdr *ph, const unsigned char *pb, const PrepLayout &pl,
                                                  const Geo &g, int i, int j, int gd, Emit emit) {
    // kAll: also hand over the strategies that do not apply (only the kept stage-cost
    // tensor wants them; the per-position loads skip them anyway)
    const int K = ph->K, lu = ph->lu;
    const uint32_t *ss = reinterpret_cast<const uint32_t *>(pb + pl.ssort);
    const uint32_t *sg = reinterpret_cast<const uint32_t *>(pb + pl.sgrp);
    const uint32_t *sd = reinterpret_cast<const uint32_t *>(pb + pl.sgd);
    const int g0 = int(sd[gd]), g1 = int(sd[gd + 1]);   // its strategy groups
    const int q0 = int(sg[g0]), q1 = int(sg[g1]);       // its strategies
    const uint32_t c0 = ss[q0];
    const int lt = c0 & 15, lcp = (c0 >> 4) & 15;
    const int ltc = lt + lcp;
    StageSums u;
    const bool stage = pair_sums(ph, pb, pl, g, i, j, u);
    if (!stage || ltc - lu > K - 1) {
        if (kAll)
            for (int m = 0; m < K; m++)
                for (int q = q0; q < q1; q++) emit(m, int(ss[q] >> 16), int64_t(-1), 0);
        return;
    }
    const int64_t Fl = u.v[kFl], Pd = u.v[kPd], Pe = u.v[kPe], Ao = u.v[kAo], Aw = u.v[kAw], A2 = u.v[kA2];
    const int64_t nM = u.v[kNm], nL = u.nL;
    const Net net{ph};
    // width-independent terms of the dense group: compute per recompute choice, the TP and
    // CP collectives inside one replica, weights, activations and stash
    const int64_t tpcp = net.coll(2, lt, ph->tier_log[lt], 4 * up_shift(Ao, lcp), 4 * nL) +
                         net.coll(1, lcp, ph->tier_log[ltc], 4 * up_shift(Ao, lt), 4 * nL);
    const int64_t cmp0 = int64_t(divide_up(uint64_t(up_shift(Fl * 3, ltc)), uint64_t(ph->R), ph->Rdiv)) + tpcp;
    const int64_t cmp1 = int64_t(divide_up(uint64_t(up_shift(Fl * 4, ltc)), uint64_t(ph->R), ph->Rdiv)) + tpcp;
    const int64_t Wd = up_shift(Pd, lt);
    const int64_t act0 = up_shift(Aw, ltc), act1 = up_shift(u.awmax, ltc);
    const int64_t st0 = act0, st1 = up_shift(reinterpret_cast<const int64_t *>(pb + pl.ain)[i], ltc);
    const float inv0 = st0 > 0 ? 1.0f / float(st0) : 0.0f, inv1 = st1 > 0 ? 1.0f / float(st1) : 0.0f;
    const int64_t full0 = int64_t(ph->P - 1) * st0, full1 = int64_t(ph->P - 1) * st1;
    const int64_t opt = ph->opt, budget = ph->budget, M = ph->M;
    const int P = ph->P;
    const bool gpipe = ph->schedule == 1;
    const int64_t owd = opt * Wd;
    // the expert AllToAlls of each strategy group (they do not depend on the width)
    int64_t epv[16];
    for (int gi = g0; gi < g1 && gi - g0 < 16; gi++) {
        const int le = (ss[sg[gi]] >> 8) & 15;
        epv[gi - g0] = net.coll(1, le, ph->tier_log[ltc + le], 4 * up_shift(A2, ltc), 4 * nM);
    }
    // strategy groups holding the whole (z, r) grid in order (eight members): their
    // members are evaluated unrolled, every select folded
    uint32_t grids = 0;
    for (int gi = g0; gi < g1 && gi - g0 < 32; gi++) {
        const int qa = int(sg[gi]), qb = int(sg[gi + 1]);
        bool grid = qb - qa == 8;
        for (int k = 0; k < 8 && grid; k++) grid = ((ss[qa + k] >> 12) & 7) == uint32_t(k >> 1 | (k & 1) << 2);
        grids |= uint32_t(grid) << (gi - g0);
    }
    for (int m = 0; m < K; m++) {
        const int lq = lu + m - ltc;
        if (lq < 0) {
            if (kAll)
                for (int q = q0; q < q1; q++) emit(m, int(ss[q] >> 16), int64_t(-1), 0);
            continue;
        }
        const int tk = ph->tier_log[lu + m];
        int64_t D1, D2;
        net.coll12(lq, tk, Wd, nL, D1, D2);
        const int64_t wdq = up_shift(Wd, lq), owdq = up_shift(owd, lq);
        for (int gi = g0; gi < g1; gi++) {
            const int qa = int(sg[gi]), qb = int(sg[gi + 1]);
            const int le = (ss[qa] >> 8) & 15;
            const int lqe = lq - le;
            if (lqe < 0 || (le > 0 && nM == 0)) {
                if (kAll)
                    for (int q = qa; q < qb; q++) emit(m, int(ss[q] >> 16), int64_t(-1), 0);
                continue;
            }
            // the strategy group's expert degree: its weights, AllToAlls and expert sync
            const int64_t We = up_shift(Pe, lt + le);
            const int64_t full = Wd + We;
            const int64_t sh = wdq + up_shift(We, lqe);
            const int64_t osh = owdq + up_shift(opt * We, lqe);
            const int64_t sz0 = 2 * full + opt * full, sz1 = 2 * full + osh, sz2 = full + sh + osh, sz3 = 2 * sh + osh;
            // Memory shrinks as the ZeRO stage grows (sz0 >= sz1 >= sz2 >= sz3: each of
            // weights, gradients and optimizer states is at most its unsharded size), so
            // when even ZeRO-3 with the smaller activation exceeds the budget, no member
            // fits the first position and none reaches a per-position load: the group
            // is not priced (only the kept cost tensor wants its words)
            if (!kAll && sz3 + (act0 < act1 ? act0 : act1) > budget) continue;
            const int64_t ep = gi - g0 < 16 ? epv[gi - g0]
                                            : net.coll(1, le, ph->tier_log[ltc + le], 4 * up_shift(A2, ltc), 4 * nM);
            int64_t E1, E2;
            net.coll12(lqe, tk, We, nM, E1, E2);
            const int64_t S1 = D1 + E1, S2 = D2 + E2;
            // the syncs amortised over M: ceil(S2 / M), and from S1 = qM + rm both
            // ceil(S1 / M) = q + (rm > 0) and ceil(2 S1 / M) = 2q + ceil(2 rm / M)
            const int64_t dM0 = int64_t(divide_up(uint64_t(S2), uint64_t(M), ph->Mdiv));       // z = 0
            const int64_t q1M = int64_t(divide(uint64_t(S1), ph->Mdiv)), rm = S1 - q1M * M;
            const int64_t dM3 = q1M + (rm > 0);                                                  // z = 3
            const int64_t dM12 = 2 * q1M + (2 * rm > M ? 2 : rm > 0 ? 1 : 0);                 // z = 1, 2
            const int64_t r0 = cmp0 + ep, r1 = cmp1 + ep;
            const int64_t t00 = up_shift(r0, lq), t10 = up_shift(r1, lq);            // z < 3
            const int64_t t03 = up_shift(r0 + S2, lq), t13 = up_shift(r1 + S2, lq);  // z = 3
            // one member: its time and fitting positions from its (z, r)
            auto member = [&](int q, int z, int r) {
                const int s = int(ss[q] >> 16);
                const int64_t tau = (z == 3 ? (r ? t13 : t03) : (r ? t10 : t00)) + (z == 0 ? dM0 : z == 3 ? dM3 : dM12);
                if (tau >= kCap) {
                    if (kAll) emit(m, s, int64_t(-1), 0);
                    return;
                }
                const int64_t stat = (z == 0 ? sz0 : z == 1 ? sz1 : z == 2 ? sz2 : sz3) + (r ? act1 : act0);
                const int pmax = stat > budget ? 0
                                               : fit_positions(ph, gpipe, P, budget - stat, r ? st1 : st0,
                                                               r ? full1 : full0, r ? inv1 : inv0, lq);
                emit(m, s, tau, pmax);
            };
            if (gi - g0 < 32 && (grids >> (gi - g0)) & 1) {
#pragma unroll
                for (int k = 0; k < 8; k++) member(qa + k, k >> 1, k & 1);
            } else {
                for (int q = qa; q < qb; q++) member(q, (ss[q] >> 12) & 3, (ss[q] >> 14) & 1);
            }
        }
    }
}

// The final batch-time loop and the plan of instance b, by one whole warp; `walk`
// is 64 ints of shared scratch for the warp (stage q -> (i | j << 8 | m << 16 |
// c' << 20, p)).
__device__ __forceinline__ void backtrack_warp_body(const PassArgs &a, int b, int *walk) {
    const int lane = threadIdx.x & 31;
    const PrepHdr *ph = prep_hdr(a, b);
    nest_plan_header *hdr = reinterpret_cast<nest_plan_header *>(a.plans_out + int64_t(b) * a.plan_stride);
    nest_stage *st = reinterpret_cast<nest_stage *>(hdr + 1);
    int status = ph->status;
    const Geo &g = a.g;
    const int64_t row_cells = int64_t(g.Cmax) * g.Dpad;
    const int64_t pos_cells = int64_t(g.Nmax) * row_cells;
    const int64_t *dpv = reinterpret_cast<const int64_t *>(a.ws + a.w.dpv) + int64_t(b) * a.w.dp_stride;
    const uint32_t *dpa = reinterpret_cast<const uint32_t *>(a.ws + a.w.dpa) + int64_t(b) * a.w.dp_stride;
    const uint64_t *loads = reinterpret_cast<const uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride;

    // smallest (t_batch, p); t_batch < 2^61
    long long bt = -1;
    int bp = 0;
    if (status == NEST_SOLVED) {
        const int L = ph->L, P = ph->P, Du = ph->Du;
        for (int p = lane + 1; p <= P && p <= L; p += 32) {
            const int64_t v = dpv[int64_t(p - 1) * pos_cells + Du];  // (i = 0, c = 0, d = Du)
            if (v < kCap) {
                const long long t = (long long)(v) * (long long)(ph->M + p - 1);
                if (bp == 0 || t < bt) {
                    bt = t;
                    bp = p;
                }
            }
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        const long long ot = __shfl_xor_sync(0xffffffffu, bt, off);
        const int op = __shfl_xor_sync(0xffffffffu, bp, off);
        if (op != 0 && (bp == 0 || ot < bt || (ot == bt && op < bp))) {
            bt = ot;
            bp = op;
        }
    }
    if (status == NEST_SOLVED && bp == 0) status = NEST_INFEASIBLE;
    if (status != NEST_SOLVED) {
        if (lane == 0) {
            hdr->status = status;
            hdr->n_stages = 0;
            hdr->t_batch = -1;
            hdr->bottleneck = -1;
            a.costs_out[b] = -1;
        }
        return;
    }
    // lane 0 follows the argument fields (a chain of dependent reads); the stages'
    // strategies are looked up afterwards by one lane each
    const int L = ph->L;
    int n = 0;
    if (lane == 0) {
        int i = 0, p = bp, c = 0, d = ph->Du;
        while (i < L && p >= 1 && n < g.Pcap) {
            const uint32_t arg = dpa[int64_t(p - 1) * pos_cells + int64_t(i) * row_cells + int64_t(c) * g.Dpad + d];
            const int j = int((arg >> 8) & 0xFF), m = int((arg >> 4) & 0xF), c2 = int(arg & 0xF);
            if (j <= i || j > L || m >= ph->K || (1 << m) > d || c2 >= ph->C) break;  // not for a solved cell
            walk[2 * n] = i | j << 8 | m << 16 | c2 << 20;
            walk[2 * n + 1] = p;
            n++;
            d -= 1 << m;
            p -= 1;
            c = c2;
            i = j;
        }
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    __syncwarp();
    if (lane < n) {
        const int w = walk[2 * lane], p = walk[2 * lane + 1];
        const int i = w & 0xFF, j = (w >> 8) & 0xFF, m = (w >> 16) & 0xF, c2 = (w >> 20) & 0xF;
        const uint64_t lw = loads[int64_t(p - 1) * g.NP * g.Kpad + (row_offset(i, L) + (j - i - 1)) * g.Kpad + m];
        st[lane].i = int16_t(i);
        st[lane].j = int16_t(j);
        st[lane].s = int16_t(lw & 0xFFFF);
        st[lane].c_next = int8_t(j < L ? c2 : -1);
        st[lane].reserved = 0;
        st[lane].k = ph->unit << m;
        st[lane].reserved2 = 0;
        const uint64_t *um = reinterpret_cast<const uint64_t *>(reinterpret_cast<const unsigned char *>(ph) + a.pl.umask);
        st[lane].layers = um[i] & ~um[j];
    }
    if (lane == 0) {
        hdr->status = NEST_SOLVED;
        hdr->n_stages = n;
        hdr->t_batch = bt;
        hdr->bottleneck = dpv[int64_t(bp - 1) * pos_cells + ph->Du];
        a.costs_out[b] = bt;
    }
}


// The same as a called function (the backtrack kernel); the fused sweep inlines the body.
static __device__ __noinline__ void backtrack_warp(const PassArgs &a, int b, int *walk) { backtrack_warp_body(a, b, walk); }

}  // namespace nest
