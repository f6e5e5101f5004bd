// DP sweep (shared by nest_sweep.cu and the resident instantiations in
// nest_sweep_res_a.cu and nest_sweep_res_b.cu): the backward min-max recurrence of
// Nest (Network- and Memory-Aware Device Placement) §4 Eq. 3, one step per DP state
// i = L-1 .. 0 (the suffixes of a chain, or the up-sets of a layer DAG; L is the last
// state, the empty set).
//
//   dp[i][d][p][c] = min over j in (i, L], width unit * 2^m <= d units, next-link
//                    candidate c' of  max(load*(i, j, m, p) + X[i][c] + X[j][c'],
//                                         dp[j][d - 2^m][p - 1][c'])
//
// c is the candidate tier of the link into the stage starting at state i (the
// "delayed forward cost" of the not yet placed producer), c' the tier of the link to
// the next stage; a stage of width k next to a link over candidate c needs
// 2k <= G[cand c].  p counts the stages still to place (the stage's 1F1B position,
// §3.3), so load* is the per-position strategy minimum from the stage-loads pass; for
// a graph, a pair of states that is not nested has no load and is no transition.
// Cells keep the smallest packed key (v << 24) | (j << 8) | (m << 4) | c', which
// makes the argmin unique and deterministic.
//
// GB300 mapping.  One cluster of `cluster` CTAs per instance; positions p are dealt
// round-robin over the cluster (CTA r owns p = r + 1 + k * cluster).  A thread owns
// one device count d and all candidates c of that d; `jsplit` threads (adjacent
// lanes) share a cell by splitting the cut points j and combine by shuffles.
//
// Two variants:
//  - resident: every CTA keeps, in shared memory, all rows dp[j][*][p-1][*] it will
//    read for its positions p.  The owner of position p pushes each new row into the
//    shared memory of the owner of p + 1 with st.async stores that complete on a
//    per-row mbarrier, so the CTAs form a pipeline over positions and a step reads no
//    dp data from global memory.  Value words are 32-bit when exact for the instance,
//    else 64-bit; with one or two candidates the 32-bit words carry the width index
//    in their low bits (tagged: one max and one min per width).  When shared memory
//    sized for both widths would leave the batch in more waves, the sweep is two
//    launches, one per width.  At the end each cluster's
//    rank 0 picks t_batch and walks the plan (the backtrack kernel is not needed).
//  - streaming: rows dp[j > i][p-1] and the loads are staged from global memory by
//    TMA bulk copies into double-buffered shared memory, tiles of `jc` cut points,
//    with the cluster in lockstep; 64-bit words.
// Every mbarrier wait is bounded; a wait that gives up marks the instance
// NEST_TIMED_OUT, drains the copies in flight and keeps taking part in every
// cluster barrier.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "nest_stages.cuh"

namespace nest {

namespace {

constexpr int64_t kDefaultSpin = int64_t(1) << 16;   // polls of up to kSuspendNs: about a second
constexpr int kMaxThreads = 512;

// ---------------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The sources of every committed group have been read (they may be overwritten).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Orders this thread's completed async-proxy global writes (bulk copies) before its later
// generic-proxy operations (a release that other CTAs acquire).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait for the given phase of an mbarrier.  Each poll is a try_wait that
// suspends the warp in hardware for up to kSuspendNs while the phase is incomplete,
// so waiting warps do not take issue slots; after `limit` polls the wait gives up
// (limit < 0: at once).
constexpr uint32_t kSuspendNs = 20000;   // a try_wait also returns as soon as the phase completes
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase, int64_t limit) {
    if (limit < 0) return false;
    const uint32_t a = smem_addr(bar);
    for (int64_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, "
            "p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(phase), "r"(kSuspendNs)
            : "memory");
        if (done) return true;
        if (it >= limit) return false;
    }
}

// Address of `local` (a shared-memory location of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
    return r;
}

// The 32-bit words of an instance on the layered sweep (nest_layered.cu): a value v is
// held as (v << tb) | tag; values 0 .. vmax are exact, vmax + 1 ("sat") stands for any
// larger finite value, and all value bits set for no value.  Two tag modes:
//  - rank (mode 0): the tag is the rank of (m, c') among a row block's admissible pairs,
//    so one minimum orders a cut point's candidates by (v, m, c');
//  - width (mode 1): the tag is the width index m alone (fewer tag bits, more value
//    bits), and the next-link candidate c' is resolved by a compare per candidate.
// An instance takes the rank mode when its value bound (largest load plus two link
// costs, a bound of every value of its DP) fits those words, else the width mode.
struct LayWords {
    bool ok;         // the instance takes the layered sweep
    bool fits;       // its value bound is at most vmax, so no word saturates
    int mode;        // 0 = rank tags, 1 = width tags
    int tb;          // tag bits
    uint32_t nmask;  // value bits of a word
    uint32_t vmax;   // largest exact value
};

__device__ __forceinline__ LayWords lay_words(const PrepHdr *ph) {
    // rank tags: at most the pairs of the first stage, which has no input link (every
    // width up to each next-link candidate's tier)
    int E = 0;
    for (int c = 0; c < ph->C && c < 16; c++)
        if (ph->mlim[c] >= 0) E += (ph->mlim[c] < ph->K - 1 ? ph->mlim[c] : ph->K - 1) + 1;
    int tr = 1;
    while ((1 << tr) < E) tr++;
    int tw = 1;   // width tags: m = 0 .. K - 1
    while ((1 << tw) < ph->K) tw++;
    const uint64_t bound = uint64_t(ph->maxload32) + 2 * uint64_t(ph->maxX32);
    LayWords w;
    w.mode = bound <= uint64_t((1u << (32 - tr)) - 3u) ? 0 : 1;
    w.tb = w.mode == 0 ? tr : tw;
    w.nmask = ~((1u << w.tb) - 1u);
    w.vmax = (1u << (32 - w.tb)) - 3u;
    w.ok = ph->C <= 4;
    w.fits = bound <= uint64_t(w.vmax);
    return w;
}

// Whether the layered sweep leaves the instance to the 64-bit streaming sweep: more
// than four candidates, or a value beyond its words met in some cell.
__device__ __forceinline__ bool lay_leaves(const PrepHdr *ph) { return !lay_words(ph).ok || ph->lay_sat != 0; }

// ---------------------------------------------------------------------------------
// The relaxation of one cut point j for the cells (c, d) of one thread
// ---------------------------------------------------------------------------------

template <int CT>
struct Cells {
    int64_t bv[CT];   // best value per candidate c (kCap = none)
    int64_t bvx[CT];  // bv - X[i][c]: a transition improves c iff a0 < bvx and nv < bv
    uint32_t bi[CT];  // its argument (j << 8) | (m << 4) | c'
    int64_t xf[CT];   // X[i][c]

    __device__ __forceinline__ void init(const int64_t *xs_i, int nc) {
#pragma unroll
        for (int c = 0; c < CT; c++) {
            xf[c] = c < nc ? xs_i[c] : 0;
            bv[c] = kCap;
            bvx[c] = kCap - xf[c];
            bi[c] = kNoArg;
        }
    }

    __device__ __forceinline__ uint64_t key(int c) const { return (uint64_t(bv[c]) << 24) | bi[c]; }

    // Cut point j: row[c' * row_stride + x] = v(dp[j][x][p-1][c']) (kCap = none),
    // lrow[m] = load*(i, j, m, p).  Cells c run over [c_lo, nc) where the first stage
    // (c_first) has no width rule on its input link.
    __device__ __forceinline__ void relax(int j, int d, int K, int C, bool c_first, int nc, const int *cmin,
                                          const int64_t *row, int64_t row_stride, const uint64_t *lrow,
                                          const int64_t *xs_j) {
        int64_t xb[CT];
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++) xb[c2] = c2 < C ? xs_j[c2] : 0;
        for (int m = 0; m < K && (1 << m) <= d; m++) {
            const uint64_t lw = lrow[m];
            if (lw == kInf) continue;
            const int64_t tst = int64_t(lw >> 16);
            const int x = d - (1 << m);
            const int cm = cmin[m];
            const int c_lo = c_first ? 0 : cm;
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++) {
                if (c2 < cm || c2 >= C) continue;
                const int64_t nv = row[c2 * row_stride + x];
                const int64_t a0 = tst + xb[c2];
                const uint32_t idx = (uint32_t(j) << 8) | (uint32_t(m) << 4) | uint32_t(c2);
#pragma unroll
                for (int c = 0; c < CT; c++) {
                    if (c < c_lo || c >= nc) continue;
                    if (a0 < bvx[c] && nv < bv[c]) {
                        const int64_t a = a0 + xf[c];
                        const int64_t v = a > nv ? a : nv;
                        bv[c] = v;
                        bvx[c] = v - xf[c];
                        bi[c] = idx;
                    }
                }
            }
        }
    }

    // The last stage [i, L): no link out, the previous state is the base case 0.
    __device__ __forceinline__ void last_stage(int L, int d, int K, bool c_first, int nc, const int *cmin,
                                               const uint64_t *lrow) {
        for (int m = 0; m < K && (1 << m) <= d; m++) {
            const uint64_t lw = lrow[m];
            if (lw == kInf) continue;
            const int64_t tst = int64_t(lw >> 16);
            const int c_lo = c_first ? 0 : cmin[m];
#pragma unroll
            for (int c = 0; c < CT; c++) {
                if (c < c_lo || c >= nc) continue;
                const int64_t v = tst + xf[c];
                if (v < bv[c]) {
                    bv[c] = v;
                    bvx[c] = v - xf[c];
                    bi[c] = (uint32_t(L) << 8) | (uint32_t(m) << 4);
                }
            }
        }
    }
};

// Per-instance state of a sweep CTA.
struct Inst {
    int L, Du, K, C, P;
    int64_t row_cells, pos_cells, pos_loads;
    int64_t *dpv;
    uint32_t *dpa;
    const uint64_t *loads;
};

__device__ __forceinline__ Inst load_inst(const PassArgs &a, const PrepHdr *ph, int b) {
    Inst s;
    s.L = ph->L;
    s.Du = ph->Du;
    s.K = ph->K;
    s.C = ph->C;
    s.P = ph->P;
    s.row_cells = int64_t(a.g.Cmax) * a.g.Dpad;
    s.pos_cells = int64_t(a.g.Nmax) * s.row_cells;
    s.pos_loads = int64_t(a.g.NP) * a.g.Kpad;
    s.dpv = reinterpret_cast<int64_t *>(a.ws + a.w.dpv) + int64_t(b) * a.w.dp_stride;
    s.dpa = reinterpret_cast<uint32_t *>(a.ws + a.w.dpa) + int64_t(b) * a.w.dp_stride;
    s.loads = reinterpret_cast<const uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride;
    return s;
}

__device__ __forceinline__ void write_cell(const Inst &s, int Dpad, int p, int i, int c, int d, uint64_t key) {
    const int64_t at = int64_t(p - 1) * s.pos_cells + int64_t(i) * s.row_cells + int64_t(c) * Dpad + d;
    s.dpv[at] = int64_t(key >> 24);
    s.dpa[at] = uint32_t(key & 0xFFFFFF);
}

// Combine the jsplit partial minima of this thread's cells through `red`; afterwards
// the threads with js == 0 hold the final keys in keys[c].  Every thread must call it.
template <int CT>
__device__ __forceinline__ void combine(const Cells<CT> &cl, uint64_t *keys, uint64_t *red, int jsplit, int js,
                                        int tid_d, int NTd, int Cmax, int nc) {
#pragma unroll
    for (int c = 0; c < CT; c++) keys[c] = c < nc ? cl.key(c) : kInf;
    if (jsplit > 1) {
#pragma unroll
        for (int c = 0; c < CT; c++)
            if (c < nc) red[(int64_t(js) * Cmax + c) * NTd + tid_d] = keys[c];
        __syncthreads();
        if (js == 0) {
#pragma unroll
            for (int c = 0; c < CT; c++) {
                if (c >= nc) continue;
                for (int q = 1; q < jsplit; q++) {
                    const uint64_t o = red[(int64_t(q) * Cmax + c) * NTd + tid_d];
                    keys[c] = o < keys[c] ? o : keys[c];
                }
            }
        }
        __syncthreads();
    }
}

// Width rule 2k <= G[cand c]: candidate tiers increase, so the candidates that admit
// width m form a suffix c >= cmin[m].
__device__ __forceinline__ void init_cmin(int *cmin, const PrepHdr *ph, int C) {
    if (threadIdx.x < 16) {
        int c = 0;
        while (c < C && ph->mlim[c] < int(threadIdx.x)) c++;
        cmin[threadIdx.x] = c;
    }
}

// ---------------------------------------------------------------------------------
// Resident variant
// ---------------------------------------------------------------------------------

// Asynchronous store into another CTA's shared memory that completes its size in
// transaction bytes on an mbarrier of that CTA (both addresses from mapa).
__device__ __forceinline__ void st_async_remote(uint32_t addr, int64_t v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u64 [%0], %1, [%2];" ::"r"(addr), "l"(v),
                 "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_remote(uint32_t addr, uint32_t v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
                 "r"(bar)
                 : "memory");
}

// Value words of the resident variant.  `cap` marks a cell without a value, `far` an
// A entry no cell can take; every finite value stays below `cap`, and far plus any
// link cost neither overflows nor drops below cap.  32-bit words are exact when the
// largest load plus two link costs is below 2^30, which the strategy reduction and the
// prep pass record per instance; otherwise the instance uses 64-bit words.  With one or
// two candidates the 32-bit words are packed (below) when a few bits more are free.
template <typename V>
struct Word;
template <>
struct Word<uint32_t> {
    static constexpr uint32_t cap = 0x7FFFFFFFu;
    static constexpr uint32_t far = 0x80000000u;
};
template <>
struct Word<int64_t> {
    static constexpr int64_t cap = kCap;
    static constexpr int64_t far = int64_t(1) << 46;
};

// Tagged 32-bit words, taken by the instantiations for one or two candidates (KT
// widths): a value v is held as (v << tb) | m, its width index m in the tb = log2(KT)
// low bits; `cap` has every value bit set and a clear tag, `far` every bit set.  The
// maximum of two words with equal tags keeps the tag, so one unsigned minimum over the
// widths of a cut point orders its candidates by value and then by width, the order
// of the key fields, with no argument to carry alongside.  Exact while every finite
// value is at most 2^(32 - tb) - 2; an instance whose values need those bits runs with
// tb = 0 (plain values, cap = far = all ones) and finds each best's width again.
template <int KT>
struct Packed {
    static constexpr int TB = KT == 4 ? 2 : KT == 8 ? 3 : 4;
};

// The template widths and candidates a batch's geometry is instantiated for.
__host__ __device__ constexpr int kt_of(int Kmax) { return Kmax <= 4 ? 4 : Kmax <= 8 ? 8 : 16; }
__host__ __device__ constexpr int ct_of(int Cmax) { return Cmax <= 3 ? Cmax : 4; }

// Tag bits of the batch's 32-bit words: log2(KT) for one or two candidates, else 0.
__host__ __device__ constexpr int word_tag_bits(int Kmax, int Cmax) {
    return ct_of(Cmax) <= 2 ? (kt_of(Kmax) == 4 ? 2 : kt_of(Kmax) == 8 ? 3 : 4) : 0;
}

// Whether 32-bit words packed with tb tag bits hold an instance: its largest load plus
// two link costs (an upper bound of every finite value of its DP) is at most
// 2^(32 - tb) - 2 (below 2^30 with no tag).
__device__ __forceinline__ bool packed_words(const PrepHdr *ph, int tb) {
    const uint64_t lim = tb ? (uint64_t(1) << (32 - tb)) - 1 : uint64_t(1) << 30;
    return uint64_t(ph->maxload32) + 2 * uint64_t(ph->maxX32) < lim;
}

// Whether an instance takes the resident sweep's 32-bit words (tb: the batch's tag
// bits).  A chain takes them below 2^30, packed when it can and plain otherwise; a
// graph only packed (its sweep is instantiated for packed words alone).
__device__ __forceinline__ bool narrow_words(const PrepHdr *ph, int tb) {
    return packed_words(ph, ph->graph ? tb : 0);
}

// Shared-memory plan of the resident variant, in 8-byte words.
//  - H[slot][j][c'][Hpad + x] = v(dp[j][x][p-1][c']).  With 32-bit values Hpad values
//    of `cap` precede x = 0, so a width 2^m above a lane's d reads cap instead of
//    needing a test; 64-bit values (Hpad = 0) clamp x at the cap column 0 instead.
//    The lanes of a warp read different cut points j, so the row stride Hrow is chosen
//    with Hrow = dpw / s (mod 32 / s) for values of s 4-byte words and dpw device
//    counts per warp: those reads land in different banks.
//  - A[buf][slot][j][c][c'][m] = load*(i, j, m, p) + X[i][c] + X[j][c'] when both
//    links admit the width, else `far`.  With tagged 32-bit values (one or two
//    candidates) A[j] spans CT*CT*KT + 4 values, so every (c, c') run of KT widths
//    starts on 16 bytes (vector loads) and the lanes reading adjacent j start in
//    different banks; otherwise an odd number of values does the same for scalar loads.
//  - staged dp rows [2][slot][Cmax][Dpad] (int64 values, uint32 arguments).
//  - graph instances: the layer mask of every state, and per step parity the list of
//    cut points j >= i + 2 whose state lies inside state i (8-bit state indices), its
//    length and whether state i + 1 lies inside state i.
// The H and A regions are sized for whichever word width needs more, or, for a launch
// that takes only the instances of one word width (`mode` 1: 32-bit, 2: 64-bit), for
// that width alone.
struct ResPlan {
    int rowbar, X, H, A, sdv, sda, um, jl, total;  // word offsets; total = words
    int Hpad, Hcol, Hrow, Hslot;           // H strides in values of the chosen width
    int Aj, Aslot, Abuf;                   // A strides in values
    int Srow;                              // values per staged dp row: Cmax * Dpad
};

// Cap columns in front of a 32-bit row.  A warp covers 32 / jsplit consecutive device
// counts d_lo .. d_hi and reads widths up to 2^mw <= d_hi, so no lane reads further
// than 32 / jsplit - 1 columns below x = 0 (nor than 2^(Kmax-1) - 1).
__host__ __device__ inline int res_hpad(const Geo &g, int jsplit, int vbytes) {
    const int reach = (1 << (g.Kmax - 1)) < 32 / jsplit ? (1 << (g.Kmax - 1)) : 32 / jsplit;
    return vbytes == 4 ? (reach + 3) & ~3 : 0;
}

__host__ __device__ inline int res_hrow(const Geo &g, int jsplit, int vbytes) {
    const int s = vbytes / 4, mod = 32 / s, want = (32 / jsplit / s) % mod;
    int h = g.Cmax * (res_hpad(g, jsplit, vbytes) + g.Dpad);
    while (h % mod != want) h++;
    return h;
}

__host__ __device__ inline ResPlan res_plan(const Geo &g, int nown, int jsplit, int CT, int KT, int vbytes,
                                            int mode) {
    ResPlan s;
    auto up = [](int w) { return (w + 15) / 16 * 16; };   // 128-byte alignment
    int off = 0;
    s.rowbar = off;                                       // one mbarrier per (owned slot, row j)
    off = up(off + nown * g.Nmax);
    s.X = off;
    off = up(off + (g.Nmax + 1) * g.Cmax);
    s.Hpad = res_hpad(g, jsplit, vbytes);
    s.Hcol = s.Hpad + g.Dpad;
    s.Hrow = res_hrow(g, jsplit, vbytes);
    s.Hslot = g.Nmax * s.Hrow;
    const int h4 = (nown * g.Nmax * res_hrow(g, jsplit, 4) + 1) / 2, h8 = nown * g.Nmax * res_hrow(g, jsplit, 8);
    s.H = off;
    off = up(off + (mode == 1 ? h4 : mode == 2 ? h8 : h4 > h8 ? h4 : h8));
    const int aj4 = CT * CT * KT + (CT <= 2 ? 4 : 1), aj8 = CT * CT * KT + 1;
    s.Aj = vbytes == 4 ? aj4 : aj8;
    s.Aslot = (g.Nmax + 1) * s.Aj;
    s.Abuf = nown * s.Aslot;
    // two buffers of 4- or 8-byte values (in 8-byte words), sized like H
    const int a4 = nown * (g.Nmax + 1) * aj4, a8 = 2 * nown * (g.Nmax + 1) * aj8;
    s.A = off;
    off = up(off + (mode == 1 ? a4 : mode == 2 ? a8 : a4 > a8 ? a4 : a8));
    s.Srow = g.Cmax * g.Dpad;
    s.sdv = off;
    off = up(off + 2 * nown * s.Srow);
    s.sda = off;
    off = up(off + nown * s.Srow);
    s.um = off;
    off = up(off + g.Nmax + 1);
    s.jl = off;   // [2] x (count, i + 1 inside i, pad, pad) as int32, then [2][Nmax] bytes
    off = up(off + 2 + (2 * g.Nmax + 7) / 8);
    s.total = off;
    return s;
}

// Relaxation of one cut point j for the cells (c, d) of one thread: for every width
// m <= mw and next-link candidate c' the candidate is v = max(A[j][c][c'][m],
// v(dp[j][d - 2^m][p-1][c'])), tried against the running best of cell c.  Excluded
// widths read far or cap and never improve.  With NA = CT each c' has its own running
// best, visited in (c', m) order and merged by key afterwards (independent dependency
// chains); with NA = 1 one running best per cell is visited in the canonical (m, c')
// order.  Either way the first strict improvement within a running best is its
// smallest key.  `mw` is the widest width any lane of the warp admits (uniform).
template <int CT, int KT, int NA, typename V, bool PK>
__device__ __forceinline__ void relax_one(const V *Aj, const V *Hj, int Hcol, int d, uint32_t jarg, int m, int c2,
                                          int a_, V tmask, V (&bv)[CT][NA], uint32_t (&bi)[CT][NA]) {
    constexpr bool kPad = sizeof(V) == 4;   // rows padded with cap below x = 0
    constexpr bool kPk = PK;   // tagged words: the tag is the width (tmask its bits)
    const int x = kPad ? d - (1 << m) : (d - (1 << m) > 0 ? d - (1 << m) : 0);
    const V nv = kPk ? V(Hj[c2 * Hcol + x] | (V(m) & tmask)) : Hj[c2 * Hcol + x];
    const uint32_t idx = kPk ? jarg : jarg | (uint32_t(m) << 4) | uint32_t(c2);
#pragma unroll
    for (int c = 0; c < CT; c++) {
        const V av = Aj[(c * CT + c2) * KT + m];
        const V v = av > nv ? av : nv;
        // tagged words: a strictly smaller value only (tag bits set for the test)
        const bool take = (kPk ? V(v | tmask) : v) < bv[c][a_];
        bv[c][a_] = take ? v : bv[c][a_];
        bi[c][a_] = take ? idx : bi[c][a_];
    }
}

// The same for one next-link candidate c2 and exactly MT widths m < MT (every lane's
// excluded widths read far or cap): the dp values of c2 are loaded first, then each
// cell takes the minimum over its MT candidates with a tree that keeps the smaller m
// on ties, and merges it into its running best for c2.  Loads overlap and the serial
// depth is log2(MT).  On packed 32-bit words the width is the tag, so the tree is a
// plain minimum and the A words come in 16-byte loads.
template <int CT, int KT, int NA, int MT, typename V, bool PK>
__device__ __forceinline__ void relax_c2_t(const V *Aj, const V *Hj, int Hcol, int d, int c2, uint32_t jarg,
                                           V tmask, V (&bv)[CT][NA], uint32_t (&bi)[CT][NA]) {
    constexpr bool kPad = sizeof(V) == 4;   // rows padded with cap below x = 0
    if constexpr (PK) {
        // tagged words: the dp values of c2 tagged with their width, then per cell the
        // MT A words by 16-byte loads, one max per width and a tree of minima
        V nv[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) nv[m] = Hj[c2 * Hcol + d - (1 << m)] | (V(m) & tmask);
        constexpr int NV = (MT + 3) / 4;
#pragma unroll
        for (int c = 0; c < CT; c++) {
            const uint4 *a4 = reinterpret_cast<const uint4 *>(Aj + (c * CT + c2) * KT);
            V v[4 * NV];
#pragma unroll
            for (int w = 0; w < NV; w++) {
                const uint4 t = a4[w];
                v[4 * w] = t.x;
                v[4 * w + 1] = t.y;
                v[4 * w + 2] = t.z;
                v[4 * w + 3] = t.w;
            }
#pragma unroll
            for (int m = 0; m < MT; m++) v[m] = v[m] > nv[m] ? v[m] : nv[m];
#pragma unroll
            for (int w = 1; w < MT; w <<= 1)
#pragma unroll
                for (int q = 0; q + w < MT; q += 2 * w) v[q] = v[q + w] < v[q] ? v[q + w] : v[q];
            // a strictly smaller value only (a later cut point never wins a tie, whatever
            // its width): compare with the tag bits set
            const bool take = (v[0] | tmask) < bv[c][c2];
            bv[c][c2] = take ? v[0] : bv[c][c2];
            bi[c][c2] = take ? jarg : bi[c][c2];
        }
    } else {
        V nv[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) {
            const int x = kPad ? d - (1 << m) : (d - (1 << m) > 0 ? d - (1 << m) : 0);
            nv[m] = Hj[c2 * Hcol + x];
        }
#pragma unroll
        for (int c = 0; c < CT; c++) {
            V v[MT];
            int id[MT];
#pragma unroll
            for (int m = 0; m < MT; m++) {
                const V av = Aj[(c * CT + c2) * KT + m];
                v[m] = av > nv[m] ? av : nv[m];
                id[m] = m;
            }
#pragma unroll
            for (int w = 1; w < MT; w <<= 1)
#pragma unroll
                for (int q = 0; q + w < MT; q += 2 * w) {
                    const bool r = v[q + w] < v[q];   // the left holds the smaller widths
                    v[q] = r ? v[q + w] : v[q];
                    id[q] = r ? id[q + w] : id[q];
                }
            const bool take = v[0] < bv[c][c2];
            bv[c][c2] = take ? v[0] : bv[c][c2];
            bi[c][c2] = take ? jarg | (uint32_t(id[0]) << 4) | uint32_t(c2) : bi[c][c2];
        }
    }
}

// Relaxation of one cut point: for every next-link candidate c2 < C, the widths up to
// mwc[c2], the warp's widest width within c2's link tier (wider ones would read far
// in every A entry of c2, which never improves a running best).  With NA = CT each c2
// dispatches once on its (warp-uniform) width count to a fully unrolled body; with
// NA = 1 one running best per cell is visited in the canonical (m, c') order.
template <int CT, int KT, int NA, typename V, bool PK>
__device__ __forceinline__ void relax_cut(const V *Aj, const V *Hj, int Hcol, int d, int C, uint32_t jarg,
                                          const int (&mwc)[CT], V tmask, V (&bv)[CT][NA], uint32_t (&bi)[CT][NA]) {
    if constexpr (NA > 1) {
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++) {
            if (c2 >= C) break;
            switch (mwc[c2]) {
            case 0: relax_c2_t<CT, KT, NA, 1, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 1: if constexpr (KT >= 2) relax_c2_t<CT, KT, NA, 2, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 2: if constexpr (KT >= 3) relax_c2_t<CT, KT, NA, 3, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 3: if constexpr (KT >= 4) relax_c2_t<CT, KT, NA, 4, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 4: if constexpr (KT >= 5) relax_c2_t<CT, KT, NA, 5, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 5: if constexpr (KT >= 6) relax_c2_t<CT, KT, NA, 6, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 6: if constexpr (KT >= 7) relax_c2_t<CT, KT, NA, 7, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            case 7: if constexpr (KT >= 8) relax_c2_t<CT, KT, NA, 8, V, PK>(Aj, Hj, Hcol, d, c2, jarg, tmask, bv, bi); break;
            default:
                // more than 8 widths: one at a time
                for (int m = 0; m <= mwc[c2] && m < KT; m++) relax_one<CT, KT, NA, V, PK>(Aj, Hj, Hcol, d, jarg, m, c2, c2, tmask, bv, bi);
                break;
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < KT; m++) {
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++) {
                if (c2 >= C) break;
                if (m > mwc[c2]) continue;
                relax_one<CT, KT, NA, V, PK>(Aj, Hj, Hcol, d, jarg, m, c2, 0, tmask, bv, bi);
            }
        }
    }
}

// Resident variant.  Each CTA owns positions p = rank + 1 + k * cs (slots k).
//  - Slot k holds the rows dp[j][*][p_k - 1][*] pushed to it by the owner of
//    position p_k - 1: each row arrives as st.async stores that complete on that
//    row's own mbarrier, so a CTA waits only for the rows it reads and the CTAs of
//    a cluster form a pipeline over positions instead of moving in lockstep.
//  - At step i only row i + 1 of a slot is new: the cut points j >= i + 2 are relaxed
//    first, and j = i + 1 is the final item of the last slice, after a bounded wait
//    for its row, so the neighbour's push overlaps this CTA's own work.  It wins ties
//    (its key is the smaller one).
//  - The A rows of step i - 1 are built during step i into the other buffer (their
//    global loads are issued before the relaxation, so their latency is hidden).
//  - A thread owns one device count d, every candidate c of it, and a slice of the
//    cut points j.  The jsplit slices of one d are adjacent lanes of a warp and are
//    combined with shuffles, so a warp covers 32 / jsplit consecutive device counts
//    and a step has a single CTA barrier.
//  - Each step's dp rows are staged in shared memory and written to global memory
//    (for the backtrack) by bulk copies.
// The footprint is kept small so that the clusters of a whole batch are resident at
// once.
template <int CT, int KT, typename V, bool kGraph, int kTag>
__device__ __forceinline__ void resident_body(const PassArgs &a, PrepHdr *ph, int b, int rank, int64_t *sm,
                                              volatile int &abort_flag) {
    constexpr int NA = CT <= 2 ? CT : 1;   // running bests per cell
    const Geo &g = a.g;
    const int cs = a.cluster;
    const Inst s = load_inst(a, ph, b);
    const int nown = (g.Pcap + cs - 1) / cs;
    const ResPlan sp = res_plan(g, nown, a.jsplit, CT, KT, int(sizeof(V)), a.word_mode);
    uint64_t *rowbar = reinterpret_cast<uint64_t *>(sm + sp.rowbar);   // [nown][Nmax]
    V *H = reinterpret_cast<V *>(sm + sp.H);
    V *A = reinterpret_cast<V *>(sm + sp.A);
    int64_t *sdv = sm + sp.sdv;
    uint32_t *sda = reinterpret_cast<uint32_t *>(sm + sp.sda);
    uint64_t *um_s = reinterpret_cast<uint64_t *>(sm + sp.um);               // [Nmax + 1]
    int *jl_hdr = reinterpret_cast<int *>(sm + sp.jl);                       // [2][2]
    uint8_t *jl_list = reinterpret_cast<uint8_t *>(sm + sp.jl + 2);          // [2][Nmax]
    constexpr bool graph = kGraph;   // states are the up-sets of a layer DAG
    // tagged 32-bit words (kTag 1 or 2; one or two candidates): the width index rides
    // in the tb low bits of every value, so the running bests carry only the cut point
    // in bi.  With kTag 1 an instance whose values leave no room for the tag runs with
    // tb = 0 (plain values, cap = far = all ones) and finds the width of each cell's
    // best again at the end of the step; kTag 2 always has room (tb fixed)
    constexpr bool kPack = kTag != 0;
    static_assert(!kPack || (sizeof(V) == 4 && CT <= 2), "tagged words are 32-bit, one or two candidates");
    const int tb = kTag == 2 ? Packed<KT>::TB : kTag == 1 && packed_words(ph, Packed<KT>::TB) ? Packed<KT>::TB : 0;
    const V tmask = kPack ? V((1u << tb) - 1u) : V(0);
    const V cap = kPack ? V(~0u << tb) : Word<V>::cap;
    constexpr V far = kPack ? V(~0u) : Word<V>::far;

    // thread = (slot group, device count d, slice js), slices in adjacent lanes; the
    // ngrp groups of gsize threads work on different slots at the same time
    const int tid = threadIdx.x, lane = tid & 31;
    const int jsplit = a.jsplit, lgs = __ffs(jsplit) - 1;
    const int gsize = (g.Dumax * jsplit + 31) / 32 * 32, ngrp = a.threads / gsize;
    const int kg = tid / gsize, gtid = tid % gsize;
    const int js = lane & (jsplit - 1);
    const int d = (gtid >> 5) * (32 >> lgs) + (lane >> lgs) + 1;
    const int jlast = jsplit - 1;   // the slice that also takes j = i + 1
    const int64_t spin = a.spin_limit == 0 ? kDefaultSpin : a.spin_limit;
    const uint32_t row_bytes = uint32_t(sizeof(V) * s.C * (s.Du + 1));   // one pushed row
    const int L = s.L, K = s.K, C = s.C;
    const bool dlive = d <= s.Du;
    // the warp's widest width: up to d units and, after the first stage, within the
    // widest input-link tier (narrower limits are folded into A and the H padding)
    int mlog = 0;
    while (mlog + 1 < K && (2 << mlog) <= d) mlog++;
    int mlink[CT], mall_n = -1;
#pragma unroll
    for (int c = 0; c < CT; c++) {
        mlink[c] = c < C ? ph->mlim[c] : -1;
        const int mt = dlive && c < C ? (mlink[c] < mlog ? mlink[c] : mlog) : -1;
        mall_n = mt > mall_n ? mt : mall_n;
    }
    const int mw_n = __reduce_max_sync(0xFFFFFFFFu, mall_n);
    const int mw_0 = __reduce_max_sync(0xFFFFFFFFu, dlive ? mlog : -1);
    const int nown_live = rank + 1 > s.P ? 0 : (s.P - rank - 1) / cs + 1;

    // A entries (slot k, cut point j = i + 1 + r, width m) at e = (k * Nmax + r) * K + m:
    // a fixed numbering, so a thread's first entry is decoded once
    const int a_total = nown_live * g.Nmax * K;
    const int a_m = tid % K, a_r = (tid / K) % g.Nmax, a_k = tid / (K * g.Nmax);
    const bool a_have = tid < a_total;
    const uint64_t *a_src = s.loads + int64_t(a_have ? rank + a_k * cs : 0) * s.pos_loads + int64_t(a_r) * g.Kpad + a_m;
    V *a_dst = A + a_k * sp.Aslot + a_r * sp.Aj + a_m;

    const int64_t *Xg = reinterpret_cast<const int64_t *>(reinterpret_cast<const unsigned char *>(ph) + a.pl.X);
    for (int e = tid; e < (L + 1) * g.Cmax; e += blockDim.x) sm[sp.X + e] = Xg[e];
    if (graph) {
        const uint64_t *umg =
            reinterpret_cast<const uint64_t *>(reinterpret_cast<const unsigned char *>(ph) + a.pl.umask);
        for (int q = tid; q <= L; q += blockDim.x) um_s[q] = umg[q];
    }
    for (int q = tid; q < nown * g.Nmax; q += blockDim.x) mbar_init(&rowbar[q], 1);
    // the padding in front of every row: cap (never written again)
    for (int e = tid; e < nown * g.Nmax * g.Cmax * sp.Hpad; e += blockDim.x) {
        const int row = e / sp.Hpad;   // (slot, j, c') in order
        H[(row / g.Cmax) * sp.Hrow + (row % g.Cmax) * sp.Hcol + e % sp.Hpad] = cap;
    }
    if (tid == 0) abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    // arm the row barriers this CTA will receive: rows 1 .. L-1 of positions p_k - 1 >= 1
    for (int q = tid; q < nown * g.Nmax; q += blockDim.x) {
        const int k = q / g.Nmax, j = q % g.Nmax;
        const int p = rank + 1 + k * cs;
        if (p >= 2 && p <= s.P && j >= 1 && j < L) mbar_expect_tx(&rowbar[q], row_bytes);
    }

    // graph instances: the cut points j >= i + 2 of step i whose state lies inside state
    // i, compacted by one warp (ballots), and whether state i + 1 lies inside it; the
    // other pairs of states are no transition (their A entries are far)
    auto build_list = [&](int ii) {
        const uint64_t Di = um_s[ii];
        uint8_t *lst = jl_list + (ii & 1) * g.Nmax;
        int cnt = 0;
        for (int base = ii + 2; base < L; base += 32) {
            const int j = base + lane;
            const bool ok = j < L && (um_s[j] & ~Di) == 0;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
            if (ok) lst[cnt + __popc(bal & ((1u << lane) - 1u))] = uint8_t(j);
            cnt += __popc(bal);
        }
        if (lane == 0) {
            jl_hdr[(ii & 1) * 2] = cnt;
            jl_hdr[(ii & 1) * 2 + 1] = ii + 1 < L && (um_s[ii + 1] & ~Di) == 0;
        }
    };

    // A[j][c][c'][m] for a stage starting at layer i (the rows of step i): the load
    // plus both link costs when the incoming link of cell c (none for the first stage,
    // which has only c = 0) and the outgoing link c' (none for the last stage) admit m
    auto a_entry = [&](V *at, int i, int j, int m, uint64_t lw) {
#pragma unroll
        for (int c = 0; c < CT; c++) {
            const bool cin = i == 0 ? c == 0 : c < C && m <= mlink[c];
            const V xi = c < C ? V(sm[sp.X + i * g.Cmax + c]) : V(0);
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++) {
                if (c2 >= C) break;
                const bool ok = lw != kInf && cin && (j == L || m <= mlink[c2]);
                const V val = V(lw >> 16) + xi + V(sm[sp.X + j * g.Cmax + c2]);
                at[(c * CT + c2) * KT] = ok ? (kPack ? V((val << tb) | (V(m) & tmask)) : val) : far;
            }
        }
    };
    auto a_rows = [&](int i, int e0) {   // entries e0, e0 + blockDim.x, .. (decoded here)
        for (int e = e0; e < a_total; e += blockDim.x) {
            const int m = e % K, r = (e / K) % g.Nmax, k = e / (K * g.Nmax);
            if (r >= L - i) continue;
            const int p = rank + 1 + k * cs, j = i + 1 + r;
            const uint64_t lw = s.loads[int64_t(p - 1) * s.pos_loads + (row_offset(i, L) + r) * g.Kpad + m];
            a_entry(A + (i & 1) * sp.Abuf + k * sp.Aslot + j * sp.Aj + m, i, j, m, lw);
        }
    };
    a_rows(L - 1, tid);
    if (graph && tid < 32) build_list(L - 1);
    // the next position's row and barrier base in its owner's shared memory, for this
    // thread's first slot (the common case has one slot per CTA); rows of step i sit
    // i * Hrow values and i barriers further on
    const int p0 = rank + 1 + kg * cs;
    const bool has0 = kg < nown_live && p0 < s.P;
    const uint32_t rrow0 = has0 ? cluster_map(H + (p0 / cs) * sp.Hslot + sp.Hpad, uint32_t(p0 % cs)) : 0;
    const uint32_t bar0 = has0 ? cluster_map(&rowbar[(p0 / cs) * g.Nmax], uint32_t(p0 % cs)) : 0;
    cluster_sync();  // first A rows built, pads and barriers set, every CTA started: pushes may begin

    int64_t ro = row_offset(L - 1, L);   // row_offset(i, L) of the current step
    for (int i = L - 1; i >= 0; i--) {
        const int Pi = s.P < L - i ? s.P : L - i;
        const int mw = i > 0 ? mw_n : mw_0;
        int mwc[CT];   // widest width per next-link candidate (its tier's limit)
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++) mwc[c2] = c2 < C ? (mlink[c2] < mw ? mlink[c2] : mw) : -1;
        // the loads of step i - 1, fetched now and stored after the relaxation
        ro -= L - i + 1;   // row_offset(i - 1, L)
        const bool a_mine = a_have && i > 0 && a_r <= L - i;
        const uint64_t pre = a_mine ? a_src[ro * g.Kpad] : kInf;
        // cut points j >= i + 2 dealt round-robin over the slices; j = i + 1 (whose row
        // arrives last) is the final item of the last slice.  A graph instance takes only
        // the states inside state i (its list for this step)
        const int n = graph ? jl_hdr[(i & 1) * 2] : (L - i - 2 > 0 ? L - i - 2 : 0);
        const bool take1 = !graph || jl_hdr[(i & 1) * 2 + 1] != 0;
        const uint8_t *jlst = jl_list + (i & 1) * g.Nmax;
        const int cnt = n > js ? (n - js + jsplit - 1) >> lgs : 0;
        const int items = cnt + (js == jlast ? 1 : 0);

        for (int k = kg; k < nown_live; k += ngrp) {
            const int p = rank + 1 + k * cs;
            V bv[CT][NA];   // running bests
            uint32_t bi[CT][NA];
            V bv_keep[CT][NA];   // packed words: the bests before the bump of the last item
#pragma unroll
            for (int c = 0; c < CT; c++)
#pragma unroll
                for (int q = 0; q < NA; q++) {
                    bv[c][q] = cap;
                    bi[c][q] = kNoArg;
                }
            const V *Ak = A + (i & 1) * sp.Abuf + k * sp.Aslot;
            const V *Hk = H + k * sp.Hslot + sp.Hpad;
            if (p == 1) {
                if (js == 0) {   // the last stage [i, L): A[L][c][0][m] = load*(i, L, m, 1) + X[i][c]
#pragma unroll
                    for (int m = 0; m < KT; m++) {
                        if (m > mw) break;
                        const V *a0 = Ak + L * sp.Aj + m;
#pragma unroll
                        for (int c = 0; c < CT; c++) {
                            const V v = m <= mlog ? a0[c * CT * KT] : far;
                            const bool take = v < bv[c][0];
                            bv[c][0] = take ? v : bv[c][0];
                            bi[c][0] = take ? (uint32_t(L) << 8) | (kPack && tb ? 0u : uint32_t(m) << 4) : bi[c][0];
                        }
                    }
                }
            } else if (p <= Pi) {
                // position p first relaxes at step i = L - p: rows i + 2 .. L - 1 of
                // position p - 1 arrived during earlier steps but were not waited for yet
                if (p == L - i)
                    for (int j = L - 1; j >= i + 2; j--)
                        if (!abort_flag && !mbar_wait(&rowbar[k * g.Nmax + j], 0, spin)) abort_flag = 1;
                for (int t = 0; t < items; t++) {
                    const bool last = t == cnt;
                    const int q = js + (t << lgs);
                    const int j = last ? i + 1 : graph ? int(jlst[q]) : i + 2 + q;
                    if (last) {
                        // row i + 1 is the one the neighbour pushed last (bounded wait; later
                        // steps read it too, so the wait is kept when it is no cut point); it
                        // is the smallest cut point and wins ties, so compare against bv + 1
                        // until it has improved a running best
                        if (!abort_flag && !mbar_wait(&rowbar[k * g.Nmax + i + 1], 0, spin)) abort_flag = 1;
                        if (!take1) break;
#pragma unroll
                        for (int c = 0; c < CT; c++)
#pragma unroll
                            for (int q = 0; q < NA; q++) {
                                if constexpr (kPack) {   // value + 1 with a clear tag: equal values win
                                    bv_keep[c][q] = bv[c][q];
                                    bv[c][q] = bv[c][q] < cap ? V((bv[c][q] | tmask) + 1) : bv[c][q];
                                } else {
                                    bv[c][q] += bv[c][q] < cap ? 1 : 0;
                                }
                            }
                    }
                    relax_cut<CT, KT, NA, V, kPack>(Ak + j * sp.Aj, Hk + j * sp.Hrow, sp.Hcol, d, C, uint32_t(j) << 8, mwc,
                                                    tmask, bv, bi);
                    if (last) {
#pragma unroll
                        for (int c = 0; c < CT; c++)
#pragma unroll
                            for (int q = 0; q < NA; q++) {   // bumped and not improved: undo
                                if constexpr (kPack)
                                    bv[c][q] = int(bi[c][q] >> 8) == i + 1 ? bv[c][q] : bv_keep[c][q];
                                else
                                    bv[c][q] -= bi[c][q] != kNoArg && int(bi[c][q] >> 8) != i + 1 ? 1 : 0;
                            }
                    }
                }
            }
            // merge the running bests by key, then the slices of the same d (lanes)
            uint64_t key[CT];
#pragma unroll
            for (int c = 0; c < CT; c++) {
                key[c] = kInf;
#pragma unroll
                for (int q = 0; q < NA; q++) {
                    uint64_t kq;
                    if constexpr (kPack) {
                        // the width: the tag; with tb = 0 the last stage recorded it and a
                        // cut point's best finds it again, the smallest width of that cut
                        // point that reaches the value
                        uint32_t mm = tb ? uint32_t(bv[c][q] & tmask) : (bi[c][q] >> 4) & 15u;
                        if (!tb && p > 1 && bv[c][q] < cap) {
                            const int jw = int(bi[c][q] >> 8);
                            const V *aw = Ak + jw * sp.Aj + (c * CT + q) * KT;
                            const V *hw = Hk + jw * sp.Hrow + q * sp.Hcol + d;
#pragma unroll
                            for (int m = KT - 1; m >= 0; m--) {
                                if (m > mwc[q]) continue;
                                const V hx = hw[-(1 << m)];
                                mm = (aw[m] > hx ? aw[m] : hx) == bv[c][q] ? uint32_t(m) : mm;
                            }
                        }
                        kq = bv[c][q] < cap ? (uint64_t(bv[c][q] >> tb) << 24) | (bi[c][q] & 0xFFFF00u) | (mm << 4) |
                                                  uint32_t(q)
                                            : kInf;
                    } else {
                        kq = bv[c][q] < cap ? (uint64_t(bv[c][q]) << 24) | bi[c][q] : kInf;
                    }
                    key[c] = kq < key[c] ? kq : key[c];
                }
            }
            __syncwarp();
            for (int o = 1; o < jsplit; o <<= 1)
#pragma unroll
                for (int c = 0; c < CT; c++) {
                    const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, key[c], o);
                    key[c] = other < key[c] ? other : key[c];
                }
            // slice js finishes the cells c = js, js + jsplit, ..: the value goes to the
            // owner of position p + 1 (its slot p / cs, row i), value and argument to the
            // staged dp row that is copied to global memory after the step
            const bool push = p < s.P && i > 0;
            uint32_t rrow = 0, bar = 0;
            if (push && k == kg) {
                rrow = rrow0 + uint32_t(i * sp.Hrow * int(sizeof(V)));
                bar = bar0 + uint32_t(8 * i);
            } else if (push) {
                const uint32_t crank = uint32_t(p % cs);
                rrow = cluster_map(H + (p / cs) * sp.Hslot + i * sp.Hrow + sp.Hpad, crank);
                bar = cluster_map(&rowbar[(p / cs) * g.Nmax + i], crank);
            }
            const int so = ((i & 1) * nown + k) * sp.Srow;
            const bool aborted = abort_flag;
#pragma unroll
            for (int c = 0; c < CT; c++) {
                if (c >= C || (c & (jsplit - 1)) != js) continue;
                const uint64_t kc = aborted ? kInf : key[c];
                const int at = c * g.Dpad + d, ht = c * sp.Hcol + d;
                if (dlive) {
                    sdv[so + at] = int64_t(kc >> 24);
                    sda[so + at] = uint32_t(kc & 0xFFFFFF);
                    if (push)
                        st_async_remote(rrow + uint32_t(ht * sizeof(V)), kc == kInf ? cap : V(V(kc >> 24) << tb), bar);
                }
                if (d == 1) {
                    sdv[so + at - 1] = kCap;
                    sda[so + at - 1] = kNoArg;
                    if (push) st_async_remote(rrow + uint32_t((ht - 1) * sizeof(V)), cap, bar);
                }
            }
        }
        // the A rows of step i - 1, into the other buffer (last read at step i + 1), after
        // this step's pushes (which the neighbour is waiting for)
        if (a_mine) a_entry(a_dst + ((i - 1) & 1) * sp.Abuf + i * sp.Aj, i - 1, i + a_r, a_m, pre);
        if (i > 0 && a_total > int(blockDim.x)) a_rows(i - 1, tid + blockDim.x);
        if (graph && i > 0 && tid < 32) build_list(i - 1);
        // the staged rows of step i go to global memory by bulk copies; those of step
        // i + 1 have been read by now (their buffer is written again at step i - 1)
        fence_proxy_async();
        if (tid == 0) bulk_wait_read();
        __syncthreads();
        if (tid == 0 && nown_live > 0) {
            for (int k = 0; k < nown_live; k++) {
                const int p = rank + 1 + k * cs;
                const int so = ((i & 1) * nown + k) * sp.Srow;
                const int64_t at = int64_t(p - 1) * s.pos_cells + int64_t(i) * s.row_cells;
                bulk_s2g(s.dpv + at, sdv + so, uint32_t(8 * C * g.Dpad));
                bulk_s2g(s.dpa + at, sda + so, uint32_t(4 * C * g.Dpad));
            }
            bulk_commit();
        }
    }
    if (tid == 0) {
        bulk_wait_all();
        fence_proxy_async_global();   // the dp rows are read by rank 0's plan walk
    }
    // every row pushed to this CTA has landed before it may exit (bounded waits)
    if (tid == 0) {
        for (int k = 0; k < nown; k++) {
            const int p = rank + 1 + k * cs;
            if (p < 2 || p > s.P) continue;
            for (int j = 1; j < L; j++) mbar_wait(&rowbar[k * g.Nmax + j], 0, kDefaultSpin);
        }
    }
    if (tid == 0 && abort_flag) ph->status = NEST_TIMED_OUT;   // before the barrier: rank 0 reads it
    cluster_sync();
}

// Each (word kind, graph) variant of the body: a called function for up to two
// candidates, so that every variant gets its own register allocation (measured: 4 %
// faster on the dense workload than all variants inlined into the kernel), inlined for
// three or four (called, those spill).
template <int CT, int KT, typename V, bool kGraph, int kTag>
__device__ __noinline__ void resident_body_call(const PassArgs &a, PrepHdr *ph, int b, int rank, int64_t *sm,
                                                volatile int &abort_flag) {
    resident_body<CT, KT, V, kGraph, kTag>(a, ph, b, rank, sm, abort_flag);
}

// The body of an instance: 32-bit words are tagged for one or two candidates, with the
// tag width chosen per instance for chains and fixed for graphs (measured: a third
// 32-bit body in the kernel, even one never called, slows the others by 4 %).
template <int CT, int KT, typename V>
__device__ __forceinline__ void run_body(const PassArgs &a, PrepHdr *ph, int b, int rank, int64_t *sm,
                                         volatile int &abort_flag) {
    constexpr bool tag = sizeof(V) == 4 && CT <= 2;
    if constexpr (CT <= 2) {
        if (ph->graph)
            resident_body_call<CT, KT, V, true, tag ? 2 : 0>(a, ph, b, rank, sm, abort_flag);
        else
            resident_body_call<CT, KT, V, false, tag ? 1 : 0>(a, ph, b, rank, sm, abort_flag);
    } else {
        if (ph->graph)
            resident_body<CT, KT, V, true, 0>(a, ph, b, rank, sm, abort_flag);
        else
            resident_body<CT, KT, V, false, 0>(a, ph, b, rank, sm, abort_flag);
    }
}

// MAXT: the largest CTA the instantiation serves.  512 threads at 2 CTAs per SM leave
// 64 registers per thread; CTAs of up to 256 threads with one or two candidates get an
// instantiation for 3 CTAs per SM, which leaves 85 (measured: 3 % faster on the dense
// workload, whose 256-thread CTAs no longer spill).
template <int CT, int KT, int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 256 ? 3 : 2) sweep_resident_kernel(PassArgs a) {
    extern __shared__ __align__(128) int64_t sm[];
    __shared__ volatile int abort_flag;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x / a.cluster;
    const int rank = int(cluster_rank());
    PrepHdr *ph = prep_hdr(a, b);
    __shared__ int walk[64];   // the plan walk's scratch
    if (ph->status != NEST_SOLVED) {   // uniform over the cluster
        // the plan header of an instance that is not solved; the 64-bit launch of a split
        // sweep leaves it to the first launch
        if (a.fuse_walk && a.word_mode != 2 && rank == 0 && threadIdx.x < 32) backtrack_warp_body(a, b, walk);
        return;
    }
    // the word width is uniform over the cluster too: every CTA reads the same header;
    // a launch for one width leaves the other width's instances to its companion launch.
    // With one or two candidates the 32-bit words carry a width tag
    const bool narrow = narrow_words(ph, CT <= 2 ? Packed<KT>::TB : 0);
    if ((a.word_mode == 1 && !narrow) || (a.word_mode == 2 && narrow)) return;
    if (!narrow)
        run_body<CT, KT, int64_t>(a, ph, b, rank, sm, abort_flag);
    else
        run_body<CT, KT, uint32_t>(a, ph, b, rank, sm, abort_flag);
    // the final reduction and the plan, by one warp of rank 0, once every CTA of the
    // cluster has written its dp rows (the cluster barrier at the end of the sweep);
    // other clusters' sweeps hide it.  Its indices are read again here so that nothing
    // stays live across the body (which would take registers from it).
    if (a.fuse_walk && cluster_rank() == 0 && threadIdx.x < 32) backtrack_warp_body(a, int(blockIdx.x) / a.cluster, walk);
}

template <typename Kern>
int set_attributes(Kern fn, size_t smem, int cluster, const char *what) {
    if (int rc = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)), what))
        return rc;
    if (cluster > 8)
        return cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1), what);
    return NEST_OK;
}

inline cudaLaunchConfig_t cluster_config(int n, int cluster, int threads, size_t smem, void *stream,
                                  cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(n * cluster), 1, 1);
    cfg.blockDim = dim3(unsigned(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <typename Kern>
int launch_cluster(Kern fn, const PassArgs &a, void *stream, size_t smem, const char *what) {
    if (int rc = set_attributes(fn, smem, a.cluster, what)) return rc;
    return launch_kernel(fn, dim3(unsigned(a.n * a.cluster)), dim3(unsigned(a.threads)), smem, stream, a.cluster, what,
                         a);
}

// The resident variant is instantiated for 1, 2, 3 or 4 candidates and KT = 4, 8 or 16 widths.

template <int CT, int KT, int MAXT>
int resident_capacity_b(int cluster, int threads, size_t smem) {
    if (set_attributes(sweep_resident_kernel<CT, KT, MAXT>, smem, cluster, "resident occupancy") != NEST_OK) return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(1, cluster, threads, smem, nullptr, attr);
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, sweep_resident_kernel<CT, KT, MAXT>, &cfg) != cudaSuccess) {
        cudaGetLastError();   // clear the error of an unsupported shape
        return 0;
    }
    return num;
}

// The instantiation a CTA of `threads` threads runs (see sweep_resident_kernel).
template <int CT>
constexpr bool small_bounds_ok() { return CT <= 2; }

template <int CT, int KT>
int resident_capacity(int cluster, int threads, size_t smem) {
    if constexpr (small_bounds_ok<CT>())
        if (threads <= 256) return resident_capacity_b<CT, KT, 256>(cluster, threads, smem);
    return resident_capacity_b<CT, KT, kMaxThreads>(cluster, threads, smem);
}

template <int CT>
int resident_capacity_kt(int KT, int cluster, int threads, size_t smem) {
    if (KT == 4) return resident_capacity<CT, 4>(cluster, threads, smem);
    if (KT == 8) return resident_capacity<CT, 8>(cluster, threads, smem);
    return resident_capacity<CT, 16>(cluster, threads, smem);
}


template <int CT, int KT>
int launch_resident(const PassArgs &a, void *stream) {
    if (a.cluster < 2 && a.g.Pcap > 1) return NEST_E_LIMITS;   // pushes need a peer CTA
    const size_t smem = size_t(sweep_resident_smem_bytes(a.g, a.cluster, a.jsplit, a.threads, a.word_mode));
    if constexpr (small_bounds_ok<CT>())
        if (a.threads <= 256)
            return launch_cluster(sweep_resident_kernel<CT, KT, 256>, a, stream, smem, "sweep (resident) launch");
    return launch_cluster(sweep_resident_kernel<CT, KT, kMaxThreads>, a, stream, smem, "sweep (resident) launch");
}

template <int CT>
int launch_resident_kt(const PassArgs &a, void *stream) {
    const int KT = kt_of(a.g.Kmax);
    if (KT == 4) return launch_resident<CT, 4>(a, stream);
    if (KT == 8) return launch_resident<CT, 8>(a, stream);
    return launch_resident<CT, 16>(a, stream);
}

}  // namespace

// The resident variant's instantiations, one translation unit per pair of candidate
// counts (compiled side by side): the clusters of one wave for `threads`-thread CTAs
// with `smem` bytes of shared memory, and the launch.
int resident_capacity_12(int CT, int KT, int cluster, int threads, size_t smem);
int resident_capacity_34(int CT, int KT, int cluster, int threads, size_t smem);
int launch_resident_12(int CT, const PassArgs &a, void *stream);
int launch_resident_34(int CT, const PassArgs &a, void *stream);

}  // namespace nest
