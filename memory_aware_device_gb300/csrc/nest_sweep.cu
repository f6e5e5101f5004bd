// DP sweep: the backward min-max recurrence of Nest (Network- and Memory-Aware
// Device Placement) §4 Eq. 3, one step per start layer i = L-1 .. 0.
//
//   dp[i][d][p][c] = min over j in (i, L], width unit * 2^m <= d units, next-link
//                    candidate c' of  max(load*(i, j, m, p) + X[i][c] + X[j][c'],
//                                         dp[j][d - 2^m][p - 1][c'])
//
// c is the candidate tier of the link into the stage starting at i (the "delayed
// forward cost" of the not yet placed producer), c' the tier of the link to the
// next stage; a stage of width k next to a link over candidate c needs
// 2k <= G[cand c].  p counts stages of the suffix (the stage's 1F1B position,
// §3.3), so load* is the per-position strategy minimum from the reduction pass.
// Cells keep the smallest packed key (v << 24) | (j << 8) | (m << 4) | c', which
// makes the argmin unique and deterministic.
//
// GB300 mapping.  One cluster of `cluster` CTAs per instance; positions p are
// dealt round-robin over the cluster (CTA r owns p = r + 1 + k * cluster).  A
// thread owns one device count d and all candidates c of that d; `jsplit` threads
// share a cell by splitting the cut points j and combine by a min over packed keys.
// Steps are separated by a cluster barrier (release / acquire).
//
// Two variants:
//  - resident: every CTA keeps, in shared memory, all rows dp[j][*][p-1][*] it will
//    read for its positions p.  The owner of position p pushes each new row into the
//    shared memory of the owner of p + 1 with distributed-shared-memory stores, so a
//    step reads no dp data from global memory at all; the loads of the next step are
//    prefetched by a TMA bulk copy one step ahead.  Used when the rows fit.
//  - streaming: rows dp[j > i][p-1] and the loads are staged from global memory by
//    TMA bulk copies into double-buffered shared memory, tiles of `jc` cut points.
// Every mbarrier wait is bounded; a wait that gives up marks the instance
// NEST_TIMED_OUT, drains the copies in flight and keeps taking part in every
// cluster barrier.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>

#include "nest_internal.cuh"

namespace nest {

namespace {

constexpr int64_t kDefaultSpin = int64_t(1) << 20;   // polls of up to kSuspendNs: about a second
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

// Bounded wait for the given phase of an mbarrier.  Each poll is a try_wait that
// suspends the warp in hardware for up to kSuspendNs while the phase is incomplete,
// so waiting warps do not take issue slots; after `limit` polls the wait gives up
// (limit < 0: at once).
constexpr uint32_t kSuspendNs = 1000;
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

__device__ __forceinline__ void st_cluster(uint32_t addr, int64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

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
    s.pos_cells = int64_t(a.g.Lmax) * s.row_cells;
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
// Resident variant: one thread per cell (c, d) and slice of the cut points
// ---------------------------------------------------------------------------------

// One DP cell (c, d) held by one thread.
struct Cell {
    int64_t bv;   // best value (kCap = none)
    int64_t bvx;  // bv - X[i][c]: a transition improves the cell iff a0 < bvx and nv < bv
    int64_t xf;   // X[i][c]
    uint32_t bi;  // argument (j << 8) | (m << 4) | c'

    __device__ __forceinline__ void init(int64_t x) {
        xf = x;
        bv = kCap;
        bvx = kCap - x;
        bi = kNoArg;
    }
    __device__ __forceinline__ uint64_t key() const { return (uint64_t(bv) << 24) | bi; }

    // Cut point j < L with widths m = 0 .. mtop (those this cell's input link admits):
    // lrow[m] = load*(i, j, m, p), xs_j[c'] = X[j][c'], candidate c' admits width m iff
    // m <= mlim2[c'], and row[c' * stride + x] = v(dp[j][x][p-1][c']).
    template <int CT>
    __device__ __forceinline__ void relax(int j, int d, int mtop, int C, const int *mlim2, const uint64_t *lrow,
                                          const int64_t *xs_j, const int64_t *row, int64_t stride) {
        int64_t xb[CT];
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++) xb[c2] = c2 < C ? xs_j[c2] : 0;
        for (int m = 0; m <= mtop; m++) {
            const uint64_t lw = lrow[m];
            if (lw == kInf) continue;
            const int64_t tst = int64_t(lw >> 16);
            const int x = d - (1 << m);
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++) {
                if (c2 >= C || m > mlim2[c2]) continue;
                const int64_t a0 = tst + xb[c2];
                const int64_t nv = row[c2 * stride + x];
                if (a0 < bvx && nv < bv) {
                    const int64_t a = a0 + xf;
                    bv = a > nv ? a : nv;
                    bvx = bv - xf;
                    bi = (uint32_t(j) << 8) | (uint32_t(m) << 4) | uint32_t(c2);
                }
            }
        }
    }

    // The last stage [i, L): lrow[m] = load*(i, L, m, p); the previous state is 0.
    __device__ __forceinline__ void last(int L, int mtop, const uint64_t *lrow) {
        for (int m = 0; m <= mtop; m++) {
            const uint64_t lw = lrow[m];
            if (lw == kInf) continue;
            const int64_t a0 = int64_t(lw >> 16);
            if (a0 < bvx) {
                bv = a0 + xf;
                bvx = a0;
                bi = (uint32_t(L) << 8) | (uint32_t(m) << 4);
            }
        }
    }
};

// Asynchronous 8-byte store into another CTA's shared memory that completes
// 8 transaction bytes on an mbarrier of that CTA (both addresses from mapa).
__device__ __forceinline__ void st_async_remote(uint32_t addr, int64_t v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u64 [%0], %1, [%2];" ::"r"(addr), "l"(v),
                 "r"(bar)
                 : "memory");
}

struct ResPlan {
    int64_t mbar, rowbar, X, H, Lt, red, total;
    int64_t H_slot, Lt_slot;  // bytes per owned position
};

__host__ __device__ inline ResPlan res_plan(const Geo &g, int nown, int jsplit, int threads) {
    ResPlan s;
    int64_t off = 0;
    s.mbar = off;
    off += 16;
    s.rowbar = off;                                   // one mbarrier per (owned slot, row j)
    off = align_up(off + 8 * int64_t(nown) * g.Lmax, 128);
    s.X = off;
    off = align_up(off + 8 * int64_t(g.Lmax + 1) * g.Cmax, 128);
    s.H_slot = 8 * int64_t(g.Lmax) * g.Cmax * g.Dpad;
    s.H = off;
    off = align_up(off + nown * s.H_slot, 128);
    s.Lt_slot = 8 * int64_t(g.NP) * g.Kpad;
    s.Lt = off;
    off = align_up(off + nown * s.Lt_slot, 128);
    s.red = off;
    if (jsplit > 1) off = align_up(off + 8 * int64_t(threads), 128);
    s.total = off;
    return s;
}

// Resident variant.  Each CTA owns positions p = rank + 1 + k * cs (slots k).  It
// holds in shared memory the whole loads table of its positions (one TMA bulk copy
// at the start) and, in slot k, the rows dp[j][*][p_k - 1][*] pushed to it by the
// owner of position p_k - 1: each row arrives as st.async stores that complete on
// that row's own mbarrier, so a CTA waits only for the rows it reads and the CTAs
// of a cluster form a pipeline over positions instead of moving in lockstep.  The
// footprint is kept small (three CTAs per SM) so that the clusters of a whole batch
// are resident at once.  The dp tables in global memory are written for the backtrack.
template <int CT>
__global__ void __launch_bounds__(kMaxThreads, 3) sweep_resident_kernel(PassArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int abort_flag;
    const Geo &g = a.g;
    const int cs = a.cluster;
    const int b = blockIdx.x / cs;
    const int rank = int(cluster_rank());
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;  // uniform over the cluster
    const Inst s = load_inst(a, ph, b);
    const int nown = (g.Pcap + cs - 1) / cs;
    const ResPlan sp = res_plan(g, nown, a.jsplit, a.threads);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + sp.mbar);
    uint64_t *rowbar = reinterpret_cast<uint64_t *>(smem + sp.rowbar);   // [nown][Lmax]
    int64_t *Xs = reinterpret_cast<int64_t *>(smem + sp.X);
    int64_t *H = reinterpret_cast<int64_t *>(smem + sp.H);
    uint64_t *Lt = reinterpret_cast<uint64_t *>(smem + sp.Lt);
    uint64_t *red = reinterpret_cast<uint64_t *>(smem + sp.red);

    // thread = (js, c, d): d fastest
    const int NTd = a.threads / (a.jsplit * g.Cmax);
    const int tid = threadIdx.x, tid_d = tid % NTd, c = (tid / NTd) % g.Cmax, js = tid / (NTd * g.Cmax);
    const int d = tid_d + 1;
    const int64_t spin = a.spin_limit == 0 ? kDefaultSpin : a.spin_limit;
    const int64_t Hrow = int64_t(g.Cmax) * g.Dpad;   // cells of one resident row
    const int64_t Hslot = sp.H_slot / 8;
    const int64_t Lslot = sp.Lt_slot / 8;
    const int red_stride = NTd * g.Cmax;             // threads of one js slice
    const uint32_t row_bytes = uint32_t(8 * s.C * (s.Du + 1));   // one pushed row

    int mlim2[CT];   // candidate c' admits width m iff m <= mlim2[c']
#pragma unroll
    for (int c2 = 0; c2 < CT; c2++) mlim2[c2] = c2 < s.C ? ph->mlim[c2] : -1;
    int mlog = 0;    // widths up to d units
    while (mlog + 1 < s.K && (2 << mlog) <= d) mlog++;

    const int64_t *Xg = reinterpret_cast<const int64_t *>(reinterpret_cast<const unsigned char *>(ph) + a.pl.X);
    for (int e = tid; e < (s.L + 1) * g.Cmax; e += blockDim.x) Xs[e] = Xg[e];
    for (int q = tid; q < nown * g.Lmax; q += blockDim.x) mbar_init(&rowbar[q], 1);
    const bool any = rank + 1 <= s.P;   // this CTA owns at least one position
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&mbar[0], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    // arm the row barriers this CTA will receive: rows 1 .. L-1 of positions p_k - 1 >= 1
    for (int q = tid; q < nown * g.Lmax; q += blockDim.x) {
        const int k = q / g.Lmax, j = q % g.Lmax;
        const int p = rank + 1 + k * cs;
        if (p >= 2 && p <= s.P && j >= 1 && j < s.L) mbar_expect_tx(&rowbar[q], row_bytes);
    }
    if (tid == 0 && any) {
        // the loads of every owned position, once
        const uint32_t tbytes = uint32_t(8 * (int64_t(s.L) * (s.L + 1) / 2) * g.Kpad);
        uint32_t bytes = 0;
        for (int k = 0; k < nown; k++)
            if (rank + 1 + k * cs <= s.P) bytes += tbytes;
        mbar_expect_tx(&mbar[0], bytes);
        for (int k = 0; k < nown; k++) {
            const int p = rank + 1 + k * cs;
            if (p > s.P) continue;
            bulk_g2s(Lt + int64_t(k) * Lslot, s.loads + int64_t(p - 1) * s.pos_loads, tbytes, &mbar[0]);
        }
    }
    cluster_sync();  // barriers armed and every CTA started: DSMEM pushes may begin
    bool loads_pending = any;   // the loads copy is in flight until waited for
    if (any) {
        if (mbar_wait(&mbar[0], 0, spin))
            loads_pending = false;
        else
            abort_flag = 1;
    }
    __syncwarp();

    for (int i = s.L - 1; i >= 0; i--) {
        const int Pi = s.P < s.L - i ? s.P : s.L - i;
        const int nc = i == 0 ? 1 : s.C;
        const bool live = d <= s.Du && c < nc;
        // widths this cell admits: up to d units and, after the first stage, within its link tier
        int mcell = mlog;
        if (i > 0) {
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++)
                if (c2 == c && mlim2[c2] < mcell) mcell = mlim2[c2];
        }
        const int64_t pair0 = row_offset(i, s.L);   // pair (i, j) = pair0 + j - i - 1
        for (int k = 0; k < nown; k++) {
            const int p = rank + 1 + k * cs;
            if (p > s.P) break;
            const uint64_t *lt = Lt + int64_t(k) * Lslot + (pair0 - i - 1) * g.Kpad;   // + j * Kpad
            Cell cl;
            cl.init(live ? Xs[int64_t(i) * g.Cmax + c] : 0);
            if (p >= 2 && p <= Pi) {
                // rows i+1 .. L-1 of position p - 1 must have arrived (bounded waits).  Position
                // p first relaxes at step i = L - p and then needs all of them; at every later
                // step only row i + 1 is new.
                const int jtop = p == s.L - i ? s.L - 1 : i + 1;
                for (int j = jtop; j > i; j--) {
                    if (!abort_flag && !mbar_wait(&rowbar[k * g.Lmax + j], 0, spin)) abort_flag = 1;
                }
                __syncwarp();
            }
            if (live && !abort_flag && p <= Pi) {
                if (p == 1) {
                    if (js == 0) cl.last(s.L, mcell, lt + int64_t(s.L) * g.Kpad);
                } else {
                    const int64_t *Hk = H + int64_t(k) * Hslot;
                    for (int j = i + 1 + js; j < s.L; j += a.jsplit)
                        cl.relax<CT>(j, d, mcell, s.C, mlim2, lt + int64_t(j) * g.Kpad, Xs + int64_t(j) * g.Cmax,
                                     Hk + int64_t(j) * Hrow, g.Dpad);
                }
            }
            uint64_t key = live ? cl.key() : kInf;
            if (a.jsplit > 1) {
                red[tid] = key;
                __syncthreads();
                if (js == 0)
                    for (int q = 1; q < a.jsplit; q++) {
                        const uint64_t o = red[tid + q * red_stride];
                        key = o < key ? o : key;
                    }
                __syncthreads();
            }
            if (js == 0 && c < s.C) {
                // the owner of position p + 1 keeps row i of position p in its slot p / cs
                const bool push = p < s.P && i > 0;
                const uint32_t crank = uint32_t(p % cs);
                const int64_t *dst = H + int64_t(p / cs) * Hslot + int64_t(i) * Hrow + int64_t(c) * g.Dpad;
                const uint32_t bar = push ? cluster_map(&rowbar[(p / cs) * g.Lmax + i], crank) : 0;
                if (d <= s.Du) {
                    write_cell(s, g.Dpad, p, i, c, d, key);
                    if (push) st_async_remote(cluster_map(dst + d, crank), int64_t(key >> 24), bar);
                }
                if (tid_d == 0) {
                    write_cell(s, g.Dpad, p, i, c, 0, kInf);
                    if (push) st_async_remote(cluster_map(dst, crank), kCap, bar);
                }
            }
        }
    }
    // every row pushed to this CTA has landed before it may exit (bounded waits)
    if (tid == 0) {
        for (int k = 0; k < nown; k++) {
            const int p = rank + 1 + k * cs;
            if (p < 2 || p > s.P) continue;
            for (int j = 1; j < s.L; j++) mbar_wait(&rowbar[k * g.Lmax + j], 0, kDefaultSpin);
        }
        if (loads_pending) mbar_wait(&mbar[0], 0, kDefaultSpin);
    }
    cluster_sync();
    if (tid == 0 && abort_flag) ph->status = NEST_TIMED_OUT;
}

// ---------------------------------------------------------------------------------
// Streaming variant
// ---------------------------------------------------------------------------------

struct StreamPlan {
    int64_t mbar, X, dp, bs, red, total;
    int64_t dp_tile, bs_tile;  // bytes per buffer
};

__host__ __device__ inline StreamPlan stream_plan(const Geo &g, int jc, int jsplit, int threads) {
    StreamPlan s;
    int64_t off = 0;
    s.mbar = off;
    off += 16;
    s.X = off;
    off = align_up(off + 8 * int64_t(g.Lmax + 1) * g.Cmax, 128);
    s.dp_tile = 8 * int64_t(jc) * g.Cmax * g.Dpad;
    s.bs_tile = 8 * int64_t(jc) * g.Kpad;
    s.dp = off;
    off = align_up(off + 2 * s.dp_tile, 128);
    s.bs = off;
    off = align_up(off + 2 * s.bs_tile, 128);
    s.red = off;
    if (jsplit > 1) off = align_up(off + 8 * int64_t(threads) * g.Cmax, 128);
    s.total = off;
    return s;
}

template <int CT>
__global__ void __launch_bounds__(kMaxThreads, 1) sweep_stream_kernel(PassArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int cmin[16];
    __shared__ volatile int abort_flag;
    const Geo &g = a.g;
    const int cs = a.cluster;
    const int b = blockIdx.x / cs;
    const int rank = int(cluster_rank());
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;  // uniform over the cluster
    const Inst s = load_inst(a, ph, b);
    const StreamPlan sp = stream_plan(g, a.jc, a.jsplit, a.threads);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + sp.mbar);
    int64_t *Xs = reinterpret_cast<int64_t *>(smem + sp.X);
    int64_t *dpbuf = reinterpret_cast<int64_t *>(smem + sp.dp);
    uint64_t *bsbuf = reinterpret_cast<uint64_t *>(smem + sp.bs);
    uint64_t *red = reinterpret_cast<uint64_t *>(smem + sp.red);

    const int NTd = a.threads / a.jsplit;
    const int tid = threadIdx.x, tid_d = tid % NTd, js = tid / NTd;
    const int d = tid_d + 1;
    const bool live_d = d <= s.Du;
    const int64_t spin = a.spin_limit == 0 ? kDefaultSpin : a.spin_limit;

    init_cmin(cmin, ph, s.C);
    const int64_t *Xg = reinterpret_cast<const int64_t *>(reinterpret_cast<const unsigned char *>(ph) + a.pl.X);
    for (int e = tid; e < (s.L + 1) * g.Cmax; e += blockDim.x) Xs[e] = Xg[e];
    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    uint32_t phase[2] = {0, 0};
    bool pending[2] = {false, false};   // thread 0 owns the copy pipeline state
    uint64_t keys[CT];

    for (int i = s.L - 1; i >= 0; i--) {
        const int Pi = s.P < s.L - i ? s.P : s.L - i;
        const int nc = i == 0 ? 1 : s.C;
        const int64_t *xs_i = Xs + int64_t(i) * g.Cmax;
        const int NJ = s.L - 1 - i;                     // cut points j in [i+1, L-1]
        const int nch = NJ > 0 ? (NJ + a.jc - 1) / a.jc : 0;
        // my positions with 2 <= p <= Pi are p = rank + 1 + k * cs for k >= k0
        const int k0 = rank == 0 ? 1 : 0;
        int nmy = 0;
        for (int p = rank + 1 + k0 * cs; p <= Pi; p += cs) nmy++;
        const int ntiles = nch * nmy;

        auto issue = [&](int t) {
            const int buf = t & 1;
            const int p = rank + 1 + (k0 + t / nch) * cs;
            const int j0 = i + 1 + (t % nch) * a.jc;
            const int nj = a.jc < s.L - j0 ? a.jc : s.L - j0;
            const int64_t *src_dp = s.dpv + int64_t(p - 2) * s.pos_cells + int64_t(j0) * s.row_cells;
            const uint64_t *src_bs =
                s.loads + int64_t(p - 1) * s.pos_loads + (row_offset(i, s.L) + (j0 - i - 1)) * g.Kpad;
            const uint32_t bdp = uint32_t(8 * int64_t(nj) * s.row_cells);
            const uint32_t bbs = uint32_t(8 * int64_t(nj) * g.Kpad);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(&mbar[buf], bdp + bbs);
            bulk_g2s(reinterpret_cast<unsigned char *>(dpbuf) + buf * sp.dp_tile, src_dp, bdp, &mbar[buf]);
            bulk_g2s(reinterpret_cast<unsigned char *>(bsbuf) + buf * sp.bs_tile, src_bs, bbs, &mbar[buf]);
            pending[buf] = true;
        };

        if (tid == 0 && !abort_flag) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int t = 0; t < 2 && t < ntiles; t++) issue(t);
        }

        Cells<CT> cl;
        for (int t = 0; t < ntiles; t++) {
            const int buf = t & 1;
            const int p = rank + 1 + (k0 + t / nch) * cs;
            const int chunk = t % nch;
            const int j0 = i + 1 + chunk * a.jc;
            const int nj = a.jc < s.L - j0 ? a.jc : s.L - j0;
            if (chunk == 0) cl.init(xs_i, nc);
            if (tid == 0 && !abort_flag) {
                if (mbar_wait(&mbar[buf], phase[buf], spin)) {
                    phase[buf] ^= 1;
                    pending[buf] = false;
                } else {
                    abort_flag = 1;
                }
            }
            __syncthreads();
            if (!abort_flag && live_d) {
                const int64_t *dps0 = dpbuf + buf * (sp.dp_tile / 8);
                const uint64_t *bs0 = bsbuf + buf * (sp.bs_tile / 8);
                for (int jj = js; jj < nj; jj += a.jsplit)
                    cl.relax(j0 + jj, d, s.K, s.C, i == 0, nc, cmin, dps0 + int64_t(jj) * s.row_cells, g.Dpad,
                             bs0 + int64_t(jj) * g.Kpad, Xs + int64_t(j0 + jj) * g.Cmax);
            }
            __syncthreads();  // every thread is done with this buffer
            if (tid == 0 && !abort_flag && t + 2 < ntiles) issue(t + 2);
            if (chunk == nch - 1) {
                combine<CT>(cl, keys, red, a.jsplit, js, tid_d, NTd, g.Cmax, nc);
                if (js == 0 && live_d) {
#pragma unroll
                    for (int c = 0; c < CT; c++)
                        if (c < s.C) write_cell(s, g.Dpad, p, i, c, d, c < nc ? keys[c] : kInf);
                }
                if (js == 0 && tid_d == 0)
                    for (int c = 0; c < s.C; c++) write_cell(s, g.Dpad, p, i, c, 0, kInf);
            }
        }
        // position 1 (a single last stage [i, L)) and positions beyond the suffix
        for (int p = rank + 1; p <= s.P; p += cs) {
            if (p >= 2 && p <= Pi) continue;
            if (js != 0) continue;
            if (tid_d == 0)
                for (int c = 0; c < s.C; c++) write_cell(s, g.Dpad, p, i, c, 0, kInf);
            if (!live_d) continue;
            cl.init(xs_i, nc);
            if (p == 1)
                cl.last_stage(s.L, d, s.K, i == 0, nc, cmin,
                              s.loads + (row_offset(i, s.L) + (s.L - i - 1)) * g.Kpad);
#pragma unroll
            for (int c = 0; c < CT; c++)
                if (c < s.C) write_cell(s, g.Dpad, p, i, c, d, c < nc && p == 1 ? cl.key(c) : kInf);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        cluster_sync();
    }
    if (tid == 0) {
        // drain copies still in flight (only after a wait gave up)
        for (int q = 0; q < 2; q++)
            if (pending[q]) mbar_wait(&mbar[q], phase[q], kDefaultSpin);
        if (abort_flag) ph->status = NEST_TIMED_OUT;
    }
}

template <typename Kern>
int set_attributes(Kern fn, size_t smem, int cluster, const char *what) {
    if (int rc = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)), what))
        return rc;
    if (cluster > 8)
        return cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1), what);
    return NEST_OK;
}

cudaLaunchConfig_t cluster_config(int n, int cluster, int threads, size_t smem, void *stream,
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
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(a.n, a.cluster, a.threads, smem, stream, attr);
    return cuda_status(cudaLaunchKernelEx(&cfg, fn, a), what);
}

// Clusters of the resident kernel that can be resident at once (0 if it cannot launch).
template <int CT>
int resident_capacity(int cluster, int threads, size_t smem) {
    if (set_attributes(sweep_resident_kernel<CT>, smem, cluster, "resident occupancy") != NEST_OK) return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(1, cluster, threads, smem, nullptr, attr);
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, sweep_resident_kernel<CT>, &cfg) != cudaSuccess) {
        cudaGetLastError();   // clear the sticky-free error of an unsupported shape
        return 0;
    }
    return num;
}

int resident_capacity_ct(int Cmax, int cluster, int threads, size_t smem) {
    if (Cmax <= 1) return resident_capacity<1>(cluster, threads, smem);
    if (Cmax <= 2) return resident_capacity<2>(cluster, threads, smem);
    if (Cmax <= 4) return resident_capacity<4>(cluster, threads, smem);
    if (Cmax <= 8) return resident_capacity<8>(cluster, threads, smem);
    return resident_capacity<16>(cluster, threads, smem);
}

template <int CT>
int launch_ct(const PassArgs &a, void *stream) {
    if (a.resident) {
        const size_t smem = size_t(sweep_resident_smem_bytes(a.g, a.cluster, a.jsplit, a.threads));
        return launch_cluster(sweep_resident_kernel<CT>, a, stream, smem, "sweep (resident) launch");
    }
    const size_t smem = size_t(sweep_smem_bytes(a.g, a.jc, a.jsplit, a.threads));
    return launch_cluster(sweep_stream_kernel<CT>, a, stream, smem, "sweep (streaming) launch");
}

}  // namespace

int64_t sweep_smem_bytes(const Geo &g, int jc, int jsplit, int threads) {
    return stream_plan(g, jc, jsplit, threads).total;
}

int64_t sweep_resident_smem_bytes(const Geo &g, int cluster, int jsplit, int threads) {
    const int nown = (g.Pcap + cluster - 1) / cluster;
    return res_plan(g, nown, jsplit, threads).total;
}

int sweep_configure(const Geo &g, int n, int cluster_opt, int jsplit_opt, int variant, SweepConfig &out) {
    int dev = 0, optin = 227 * 1024, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int64_t budget = 200 * 1024 < optin - 1024 ? 200 * 1024 : optin - 1024;
    auto ok_cluster = [](int c) { return c == 1 || c == 2 || c == 4 || c == 8 || c == 16; };
    auto ok_jsplit = [](int j) { return j == 1 || j == 2 || j == 4 || j == 8; };
    if ((cluster_opt && !ok_cluster(cluster_opt)) || (jsplit_opt && !ok_jsplit(jsplit_opt))) return NEST_E_INVALID;
    const int NTd = (g.Dumax + 31) / 32 * 32;

    // resident: one thread per (slice, candidate, device count); every instance's
    // cluster resident at once if possible, then the least work per thread and step
    if (variant != 2) {
        const int base = g.Cmax * NTd;
        double best = 0;
        SweepConfig pick = {};
        const int cl_list[5] = {16, 8, 4, 2, 1};
        const int js_list[4] = {8, 4, 2, 1};
        for (int ci = 0; ci < 5; ci++) {
            const int cs = cluster_opt ? cluster_opt : cl_list[ci];
            if (cs > 1 && cs > g.Pcap && !cluster_opt) continue;
            for (int ji = 0; ji < 4; ji++) {
                const int js = jsplit_opt ? jsplit_opt : js_list[ji];
                const int threads = base * js;
                if (threads > kMaxThreads) continue;
                const int64_t smem = sweep_resident_smem_bytes(g, cs, js, threads);
                if (smem > budget) continue;
                const int cap = resident_capacity_ct(g.Cmax, cs, threads, size_t(smem));
                if (std::getenv("NEST_DEBUG"))
                    std::fprintf(stderr, "nest: resident sweep cluster %d jsplit %d threads %d smem %lld: %d clusters at once\n",
                                 cs, js, threads, (long long)smem, cap);
                if (cap <= 0) continue;
                const int waves = (n + cap - 1) / cap;
                const int nown = (g.Pcap + cs - 1) / cs;
                const double score = 1.0 / (double(waves) * nown / threads);   // higher is better
                if (score > best) {
                    best = score;
                    pick = {cs, js, 0, threads, 1, waves};
                }
                if (jsplit_opt) break;
            }
            if (cluster_opt) break;
        }
        // resident only when every cluster of the pass is resident at once: otherwise the
        // streaming variant, whose CTAs need no co-scheduling, keeps the GPU fuller
        if (best > 0 && (variant == 1 || pick.resident_waves == 1)) {
            out = pick;
            if (std::getenv("NEST_DEBUG"))
                std::fprintf(stderr, "nest: sweep resident, cluster %d jsplit %d threads %d\n", pick.cluster,
                             pick.jsplit, pick.threads);
            return NEST_OK;
        }
        if (variant == 1) return NEST_E_LIMITS;
    }
    // streaming: one thread per (slice, device count) holding every candidate
    int jsplit = jsplit_opt;
    if (jsplit == 0) {
        jsplit = 1;
        while (jsplit < 8 && NTd * jsplit * 2 <= kMaxThreads) jsplit *= 2;
    }
    if (NTd * jsplit > kMaxThreads) return NEST_E_INVALID;
    int cluster = cluster_opt;
    if (cluster == 0) {
        cluster = 1;
        while (cluster < 8 && cluster * 2 <= g.Pcap && int64_t(n) * cluster * 2 <= sms) cluster *= 2;
    }
    const int threads = NTd * jsplit;
    int jc = g.Lmax > 1 ? g.Lmax - 1 : 1;
    while (jc > 1 && sweep_smem_bytes(g, jc, jsplit, threads) > budget) jc--;
    if (sweep_smem_bytes(g, jc, jsplit, threads) > budget) return NEST_E_LIMITS;
    out = {cluster, jsplit, jc, threads, 0, 1};
    return NEST_OK;
}

int launch_sweep(const PassArgs &a, void *stream) {
    if (a.g.Cmax <= 1) return launch_ct<1>(a, stream);
    if (a.g.Cmax <= 2) return launch_ct<2>(a, stream);
    if (a.g.Cmax <= 4) return launch_ct<4>(a, stream);
    if (a.g.Cmax <= 8) return launch_ct<8>(a, stream);
    return launch_ct<16>(a, stream);
}

}  // namespace nest
