// DP sweep: the streaming variant, the choice of launch shape and the launch entry.
// The recurrence, the GB300 mapping and the resident variant are described in
// nest_sweep.cuh; the resident kernels are instantiated in nest_sweep_res_a.cu and
// nest_sweep_res_b.cu.
#include "nest_sweep.cuh"

namespace nest {

namespace {

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
    off = align_up(off + 8 * int64_t(g.Nmax + 1) * g.Cmax, 128);
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
    pdl_wait();
    pdl_trigger();
    const Geo &g = a.g;
    const int cs = a.cluster;
    const int b = blockIdx.x / cs;
    const int rank = int(cluster_rank());
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;  // uniform over the cluster
    if (a.word_mode == 2 && narrow_words(ph, word_tag_bits(g.Kmax, g.Cmax))) return;   // taken by the resident launch
    if (a.word_mode == 3 && !lay_leaves(ph)) return;   // solved by the layered sweep
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

template <int CT>
int launch_ct(const PassArgs &a, void *stream) {
    const size_t smem = size_t(sweep_smem_bytes(a.g, a.jc, a.jsplit, a.threads));
    return launch_cluster(sweep_stream_kernel<CT>, a, stream, smem, "sweep (streaming) launch");
}


}  // namespace

int resident_capacity_ct(const Geo &g, int cluster, int threads, size_t smem) {
    const int KT = kt_of(g.Kmax), CT = ct_of(g.Cmax);
    if (g.Cmax > 4) return 0;
    return CT <= 2 ? resident_capacity_12(CT, KT, cluster, threads, smem)
                   : resident_capacity_34(CT, KT, cluster, threads, smem);
}

int64_t sweep_smem_bytes(const Geo &g, int jc, int jsplit, int threads) {
    return stream_plan(g, jc, jsplit, threads).total;
}

int64_t sweep_resident_smem_bytes(const Geo &g, int cluster, int jsplit, int threads, int mode) {
    const int nown = (g.Pcap + cluster - 1) / cluster;
    (void)threads;
    return 8 * int64_t(res_plan(g, nown, jsplit, ct_of(g.Cmax), kt_of(g.Kmax), 8, mode).total);
}

// Streaming shape: one thread per (slice, device count) holding every candidate.
static int stream_shape(const Geo &g, int n, int cluster_opt, int jsplit_opt, int sms, int64_t budget, SweepShape &out) {
    const int NTd = (g.Dumax + 31) / 32 * 32;
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
    int jc = g.Nmax > 1 ? g.Nmax - 1 : 1;
    while (jc > 1 && sweep_smem_bytes(g, jc, jsplit, threads) > budget) jc--;
    if (sweep_smem_bytes(g, jc, jsplit, threads) > budget) return NEST_E_LIMITS;
    out = {cluster, jsplit, jc, threads, 0, 1};
    return NEST_OK;
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
    if (variant < 0 || variant > 3) return NEST_E_INVALID;
    // layered: one launch per position over every instance's cells (up to four link
    // candidates, 32-bit tagged words); the streaming shape takes the instances whose
    // values do not fit those words
    auto layered = [&]() {
        if (g.Cmax > 4 || layered_smem_bytes(g) > budget) return int(NEST_E_LIMITS);
        SweepShape sh;
        if (int rc = stream_shape(g, n, cluster_opt, jsplit_opt, sms, budget, sh)) return rc;
        out = {sh.cluster, sh.jsplit, sh.jc, sh.threads, 0, 1, 0, {}, 1};
        return int(NEST_OK);
    };
    if (variant == 3) return layered();

    // resident: one thread per (device count, slice) holding every candidate, the
    // slices of a device count in adjacent lanes, and up to ngrp such groups per CTA
    // working on different positions.  Prefer every instance's cluster resident at
    // once, then the fewest positions per CTA (positions sharing an SM, whether in
    // turn or in parallel groups, slow each other down about as much), then larger
    // clusters, then groups of about 8 warps per 32 states, 16 at most (more warps
    // add per-step work, fewer hide less latency; a step relaxes up to one cut point
    // per later state).  `mode` sizes shared memory for both word widths (0), or for
    // a launch that takes the instances of one width only (1: 32-bit, 2: 64-bit).
    struct Pick {
        double best;
        SweepShape shape;
        int64_t ctas;   // CTAs resident at once
    };
    auto search = [&](int mode) {
        Pick r = {0.0, {}, 0};
        const int cl_list[5] = {16, 8, 4, 2, 1};
        const int js_list[4] = {8, 4, 2, 1};
        for (int ci = 0; ci < 5; ci++) {
            const int cs = cluster_opt ? cluster_opt : cl_list[ci];
            if (cs > 1 && cs > g.Pcap && !cluster_opt) continue;
            // rows are pushed to the owner of the next position with st.async, which
            // must be another CTA of the cluster: one CTA per instance only when no
            // row is pushed (a single position)
            if (cs == 1 && g.Pcap > 1) {
                if (cluster_opt) break;
                continue;
            }
            for (int ji = 0; ji < 4; ji++) {
                const int js = jsplit_opt ? jsplit_opt : js_list[ji];
                const int gsize = (g.Dumax * js + 31) / 32 * 32;
                if (gsize > kMaxThreads) continue;
                const int nown_c = (g.Pcap + cs - 1) / cs;
                const int ngrp = nown_c < kMaxThreads / gsize ? nown_c : kMaxThreads / gsize;
                const int threads = ngrp * gsize;
                const int64_t smem = sweep_resident_smem_bytes(g, cs, js, threads, mode);
                if (smem > budget) continue;
                const int cap = resident_capacity_ct(g, cs, threads, size_t(smem));
                if (std::getenv("NEST_DEBUG"))
                    std::fprintf(stderr,
                                 "nest: resident sweep words %d cluster %d jsplit %d threads %d smem %lld: %d clusters at once\n",
                                 mode, cs, js, threads, (long long)smem, cap);
                if (cap <= 0) continue;
                const int waves = (n + cap - 1) / cap;
                const int serial = (nown_c + ngrp - 1) / ngrp;
                // a pass whose CTAs fill at most half the SMs is latency-bound: the most
                // threads per instance then (measured: 16 x 32-state instances at B <= 4
                // 8 % faster with jsplit 8, at B = 8 slower)
                const bool sparse = int64_t(n) * cs * 2 <= int64_t(sms);
                const double ideal = sparse || g.Nmax >= 64 ? 512.0 : g.Nmax > 32 ? 8.0 * g.Nmax : 256.0;
                const double score = 1.0 / (double(waves) * serial * ngrp * (1.0 + (16 - cs) / 64.0) *
                                            (1.0 + std::fabs(std::log2(gsize / ideal)) / 8));
                if (score > r.best) {
                    r.best = score;
                    r.shape = {cs, js, 0, threads, 1, waves};
                    r.ctas = int64_t(cap) * cs;
                }
                if (jsplit_opt) break;
            }
            if (cluster_opt) break;
        }
        return r;
    };
    // resident when every cluster of the pass is resident at once, or when one wave
    // of clusters holds at least one CTA per SM (measured on GB300, 16-CTA clusters:
    // 64 clusters of 60 KB in 4 waves beat the streaming variant 2.7x, 16 clusters of
    // 94 KB in 2 waves 3.4x, 256 clusters in 19 waves 1.45x); with fewer CTAs per SM
    // the streaming variant, whose CTAs need no co-scheduling, keeps the GPU fuller
    auto accept = [&](const Pick &r) {
        return r.best > 0 && (variant == 1 || r.shape.resident_waves == 1 || r.ctas >= int64_t(sms));
    };
    // the library's choice between a resident shape in several waves and the layered
    // sweep: over enough states the layered launches are throughput-bound and win
    // (measured on GB300: 256 instances of 48 states, resident in waves 6.4 ms, layered
    // 4.9 ms); below that each of their launches is bound by the serial cut points of
    // its longest CTA (16 instances of 32 states: resident 0.16 ms, layered 1.7 ms)
    auto prefer_layered = [&](const SweepShape &sh) {
        return variant == 0 && sh.resident_waves >= 3 && g.Nmax >= 40 && layered() == NEST_OK;
    };
    out.split = 0;
    out.wide = {};
    if (variant != 2 && g.Cmax <= 4) {
        const Pick both = search(0);
        // rows of 32-bit words take about half the shared memory: when a launch sized
        // for them alone needs fewer waves, it takes those instances and a second launch
        // (resident if its shape fits, else streaming) takes the instances on 64-bit words
        if (!(accept(both) && both.shape.resident_waves == 1)) {
            const Pick narrow = search(1);
            if (accept(narrow) && (!accept(both) || narrow.shape.resident_waves < both.shape.resident_waves)) {
                const Pick wide = search(2);
                SweepShape ws = {};
                bool ok = wide.best > 0;
                if (ok) {
                    ws = wide.shape;
                } else if (variant != 1) {
                    ok = stream_shape(g, n, cluster_opt, jsplit_opt, sms, budget, ws) == NEST_OK;
                }
                if (ok) {
                    const SweepShape &ns = narrow.shape;
                    if (prefer_layered(ns)) return NEST_OK;
                    out = {ns.cluster, ns.jsplit, ns.jc, ns.threads, ns.resident, ns.resident_waves, 1, ws};
                    if (std::getenv("NEST_DEBUG"))
                        std::fprintf(stderr,
                                     "nest: sweep split: resident 32-bit cluster %d jsplit %d threads %d; 64-bit %s "
                                     "cluster %d jsplit %d threads %d\n",
                                     ns.cluster, ns.jsplit, ns.threads, ws.resident ? "resident" : "streaming",
                                     ws.cluster, ws.jsplit, ws.threads);
                    return NEST_OK;
                }
            }
        }
        if (accept(both)) {
            const SweepShape &p = both.shape;
            if (prefer_layered(p)) return NEST_OK;
            out = {p.cluster, p.jsplit, p.jc, p.threads, p.resident, p.resident_waves, 0, {}};
            if (std::getenv("NEST_DEBUG"))
                std::fprintf(stderr, "nest: sweep resident, cluster %d jsplit %d threads %d\n", p.cluster, p.jsplit,
                             p.threads);
            return NEST_OK;
        }
        if (variant == 1) return NEST_E_LIMITS;
    }
    if (variant == 0 && layered() == NEST_OK) return NEST_OK;
    SweepShape sh;
    if (int rc = stream_shape(g, n, cluster_opt, jsplit_opt, sms, budget, sh)) return rc;
    out = {sh.cluster, sh.jsplit, sh.jc, sh.threads, 0, 1, 0, {}, 0};
    return NEST_OK;
}

int launch_sweep(const PassArgs &a, void *stream) {
    if (a.resident) {
        const int CT = ct_of(a.g.Cmax);
        return CT <= 2 ? launch_resident_12(CT, a, stream) : launch_resident_34(CT, a, stream);
    }
    if (a.g.Cmax <= 1) return launch_ct<1>(a, stream);
    if (a.g.Cmax <= 2) return launch_ct<2>(a, stream);
    if (a.g.Cmax <= 4) return launch_ct<4>(a, stream);
    if (a.g.Cmax <= 8) return launch_ct<8>(a, stream);
    return launch_ct<16>(a, stream);
}

}  // namespace nest
