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
// GB300 mapping.  One cluster of `cluster` CTAs per instance; the positions p are
// dealt round-robin over the cluster's CTAs, so that a CTA only ever reads rows
// dp[j][*][p-1][*] written by its neighbour.  A CTA thread owns one device count d
// (and all candidates c of that d); `jsplit` threads share a cell by splitting the
// cut points j, and combine by a min over packed keys.  The rows dp[j > i][p-1]
// and the loads of (i, j, *, p) are staged into shared memory by TMA bulk copies
// (cp.async.bulk) completing on mbarriers, double-buffered over tiles of `jc` cut
// points, and reused by every (d, m, c, c') of the tile.  Steps are separated by
// a cluster barrier (release / acquire), after a proxy fence that orders this
// step's generic stores before the next step's bulk copies.  Every mbarrier wait
// is bounded; a wait that gives up marks the instance NEST_TIMED_OUT, drains the
// copies in flight and keeps taking part in the cluster barriers.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

constexpr int64_t kDefaultSpin = int64_t(1) << 26;
constexpr int kMaxThreads = 1024;

struct SmemPlan {
    int64_t mbar, X, dp, bs, red, total;
    int64_t dp_tile, bs_tile;  // bytes per buffer
};

__host__ __device__ inline SmemPlan smem_plan(const Geo &g, int jc, int jsplit, int threads) {
    SmemPlan s;
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

// Bounded wait for the given phase of an mbarrier.  limit < 0 gives up at once.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase, int64_t limit) {
    if (limit < 0) return false;
    const uint32_t a = smem_addr(bar);
    for (int64_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(phase)
            : "memory");
        if (done) return true;
        if (it >= limit) return false;
    }
}

template <int CT>
__global__ void __launch_bounds__(kMaxThreads, 1) sweep_kernel(PassArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Geo &g = a.g;
    const int cs = a.cluster;
    const int b = blockIdx.x / cs;
    const int rank = int(cluster_rank());
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;  // uniform over the cluster

    const SmemPlan sp = smem_plan(g, a.jc, a.jsplit, a.threads);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + sp.mbar);
    int64_t *Xs = reinterpret_cast<int64_t *>(smem + sp.X);
    int64_t *dpbuf = reinterpret_cast<int64_t *>(smem + sp.dp);
    uint64_t *bsbuf = reinterpret_cast<uint64_t *>(smem + sp.bs);
    uint64_t *red = reinterpret_cast<uint64_t *>(smem + sp.red);
    __shared__ int abort_flag;

    const int L = ph->L, Du = ph->Du, K = ph->K, C = ph->C, P = ph->P;
    const int NTd = a.threads / a.jsplit;
    const int tid = threadIdx.x;
    const int tid_d = tid % NTd, js = tid / NTd;
    const int d = tid_d + 1;
    const bool live_d = d <= Du;

    // Width rule 2k <= G[cand c]: candidate tiers increase, so the candidates that
    // admit width m form a suffix c >= cmin[m].
    __shared__ int cmin[16];
    if (threadIdx.x < 16) {
        int c = 0;
        while (c < C && ph->mlim[c] < int(threadIdx.x)) c++;
        cmin[threadIdx.x] = c;
    }

    const unsigned char *pb = reinterpret_cast<const unsigned char *>(ph);
    const int64_t *Xg = reinterpret_cast<const int64_t *>(pb + a.pl.X);
    for (int e = tid; e < (L + 1) * g.Cmax; e += blockDim.x) Xs[e] = Xg[e];
    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int64_t *dpv = reinterpret_cast<int64_t *>(a.ws + a.w.dpv) + int64_t(b) * a.w.dp_stride;
    uint32_t *dpa = reinterpret_cast<uint32_t *>(a.ws + a.w.dpa) + int64_t(b) * a.w.dp_stride;
    const uint64_t *loads = reinterpret_cast<const uint64_t *>(a.ws + a.w.loads) + int64_t(b) * a.w.loads_stride;
    const int64_t row_cells = int64_t(g.Cmax) * g.Dpad;                // one (p, j) row
    const int64_t pos_cells = int64_t(g.Lmax) * row_cells;            // one position p
    const int64_t pos_loads = int64_t(g.NP) * g.Kpad;
    const int64_t spin = a.spin_limit == 0 ? kDefaultSpin : a.spin_limit;

    // thread 0 owns the copy pipeline state
    uint32_t phase[2] = {0, 0};
    bool pending[2] = {false, false};

    auto write_cell = [&](int p, int i, int c, int dd, uint64_t key) {
        const int64_t at = int64_t(p - 1) * pos_cells + int64_t(i) * row_cells + int64_t(c) * g.Dpad + dd;
        dpv[at] = int64_t(key >> 24);
        dpa[at] = uint32_t(key & 0xFFFFFF);
    };

    for (int i = L - 1; i >= 0; i--) {
        const int Pi = P < L - i ? P : L - i;
        const int nc = i == 0 ? 1 : C;
        const int64_t *xf = Xs + int64_t(i) * g.Cmax;
        const int NJ = L - 1 - i;                       // cut points j in [i+1, L-1]
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
            const int nj = a.jc < L - j0 ? a.jc : L - j0;
            const int64_t *src_dp = dpv + int64_t(p - 2) * pos_cells + int64_t(j0) * row_cells;
            const uint64_t *src_bs = loads + int64_t(p - 1) * pos_loads + (row_offset(i, L) + (j0 - i - 1)) * g.Kpad;
            const uint32_t bdp = uint32_t(8 * int64_t(nj) * row_cells);
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

        int64_t bv[CT];
        uint32_t bi[CT];
        for (int t = 0; t < ntiles; t++) {
            const int buf = t & 1;
            const int p = rank + 1 + (k0 + t / nch) * cs;
            const int chunk = t % nch;
            const int j0 = i + 1 + chunk * a.jc;
            const int nj = a.jc < L - j0 ? a.jc : L - j0;
            if (chunk == 0) {
#pragma unroll
                for (int c = 0; c < CT; c++) {
                    bv[c] = kCap;
                    bi[c] = kNoArg;
                }
            }
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
                for (int jj = js; jj < nj; jj += a.jsplit) {
                    const int j = j0 + jj;
                    const int64_t *dps = dps0 + int64_t(jj) * row_cells;
                    const uint64_t *bs = bs0 + int64_t(jj) * g.Kpad;
                    const int64_t *xb = Xs + int64_t(j) * g.Cmax;
                    for (int m = 0; m < K && (1 << m) <= d; m++) {
                        const uint64_t lw = bs[m];
                        if (lw == kInf) continue;
                        const int64_t tst = int64_t(lw >> 16);
                        const int x = d - (1 << m);
                        const int cm = cmin[m];
                        const int c_lo = i == 0 ? 0 : cm;
                        for (int c2 = cm; c2 < C; c2++) {
                            const int64_t nv = dps[int64_t(c2) * g.Dpad + x];
                            const int64_t a0 = tst + xb[c2];
                            const uint32_t idx = (uint32_t(j) << 8) | (uint32_t(m) << 4) | uint32_t(c2);
#pragma unroll
                            for (int c = 0; c < CT; c++) {
                                if (c < nc && c >= c_lo) {
                                    const int64_t av = a0 + xf[c];
                                    const int64_t v = av > nv ? av : nv;
                                    if (v < bv[c]) {
                                        bv[c] = v;
                                        bi[c] = idx;
                                    }
                                }
                            }
                        }
                    }
                }
            }
            __syncthreads();  // every thread is done with this buffer
            if (tid == 0 && !abort_flag && t + 2 < ntiles) issue(t + 2);
            if (chunk == nch - 1) {
                // combine the jsplit partial cells and write row i of position p
                if (a.jsplit > 1) {
#pragma unroll
                    for (int c = 0; c < CT; c++)
                        if (c < nc) red[(int64_t(js) * g.Cmax + c) * NTd + tid_d] = (uint64_t(bv[c]) << 24) | bi[c];
                    __syncthreads();
                }
                if (js == 0 && live_d) {
#pragma unroll
                    for (int c = 0; c < CT; c++) {
                        if (c >= C) continue;
                        uint64_t key = kInf;
                        if (c < nc) {
                            key = (uint64_t(bv[c]) << 24) | bi[c];
                            for (int q = 1; q < a.jsplit; q++) {
                                const uint64_t o = red[(int64_t(q) * g.Cmax + c) * NTd + tid_d];
                                key = o < key ? o : key;
                            }
                        }
                        write_cell(p, i, c, d, key);
                    }
                }
                if (js == 0 && tid_d == 0)
                    for (int c = 0; c < C; c++) write_cell(p, i, c, 0, kInf);
                if (a.jsplit > 1) __syncthreads();
            }
        }
        // position 1 (a single last stage [i, L)) and positions beyond the suffix
        for (int p = rank + 1; p <= P; p += cs) {
            if (p >= 2 && p <= Pi) continue;
            if (js != 0) continue;
            if (tid_d == 0)
                for (int c = 0; c < C; c++) write_cell(p, i, c, 0, kInf);
            if (!live_d) continue;
            const uint64_t *lrow = loads + int64_t(p - 1) * pos_loads + (row_offset(i, L) + (L - i - 1)) * g.Kpad;
            for (int c = 0; c < C; c++) {
                uint64_t key = kInf;
                if (p == 1 && c < nc) {
                    int64_t best = kCap;
                    uint32_t arg = kNoArg;
                    for (int m = 0; m < K && (1 << m) <= d; m++) {
                        if (i > 0 && c < cmin[m]) continue;
                        const uint64_t lw = lrow[m];
                        if (lw == kInf) continue;
                        const int64_t v = int64_t(lw >> 16) + xf[c];
                        if (v < best) {
                            best = v;
                            arg = (uint32_t(L) << 8) | (uint32_t(m) << 4);
                        }
                    }
                    key = (uint64_t(best) << 24) | arg;
                }
                write_cell(p, i, c, d, key);
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        cluster_sync();
    }
    if (tid == 0) {
        // drain copies still in flight (only after a wait gave up)
        for (int buf = 0; buf < 2; buf++)
            if (pending[buf]) mbar_wait(&mbar[buf], phase[buf], kDefaultSpin);
        if (abort_flag) ph->status = NEST_TIMED_OUT;
    }
}

template <int CT>
int launch_ct(const PassArgs &a, void *stream, size_t smem) {
    auto fn = sweep_kernel<CT>;
    if (int rc = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "sweep smem attribute"))
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.n * a.cluster), 1, 1);
    cfg.blockDim = dim3(unsigned(a.threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(a.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, fn, a), "sweep launch");
}

}  // namespace

int64_t sweep_smem_bytes(const Geo &g, int jc, int jsplit, int threads) {
    return smem_plan(g, jc, jsplit, threads).total;
}

int launch_sweep(const PassArgs &a, void *stream) {
    const size_t smem = size_t(sweep_smem_bytes(a.g, a.jc, a.jsplit, a.threads));
    if (a.g.Cmax <= 1) return launch_ct<1>(a, stream, smem);
    if (a.g.Cmax <= 2) return launch_ct<2>(a, stream, smem);
    if (a.g.Cmax <= 4) return launch_ct<4>(a, stream, smem);
    if (a.g.Cmax <= 8) return launch_ct<8>(a, stream, smem);
    return launch_ct<16>(a, stream, smem);
}

}  // namespace nest
