// DP sweep by positions ("layered"): the recurrence of Nest (Network- and
// Memory-Aware Device Placement) §4 Eq. 3 evaluated one pipeline position at a time.
//
//   dp[i][d][p][c] = min over j in (i, L), width 2^m <= d, next-link candidate c' of
//                    max(load*(i, j, m, p) + X[i][c] + X[j][c'], dp[j][d - 2^m][p-1][c'])
//   dp[i][d][1][c] = min over 2^m <= d of load*(i, L, m, 1) + X[i][c]     (the last stage)
//
// Position p reads only position p - 1, so every cell (i, d, c) of one position is
// independent of the others: one launch per position computes all of them, for
// every instance of the pass, with no step barrier inside an instance.  For a fixed
// position the recurrence is a min-max product: rows (i, c), columns d and the inner
// index (j, m, c'), where the A operand load*(i, j, m, p) + X[i][c] + X[j][c'] does
// not depend on d and the B operand dp[j][d - 2^m][p-1][c'] is row (j, c') of the
// previous position shifted by 2^m.  It is tiled like a matrix product:
//  - a CTA owns RT consecutive states i and one input candidate c (a "row block"),
//    and every device count d of them; a thread owns the RT x 4 cells (i0..i0+RT-1,
//    4t+1..4t+4), so each A word is shared by 4 cells and each B word by RT;
//  - the cut points j are streamed through double-buffered shared memory: the B rows
//    (j, c') of the previous position by bulk copies (cp.async.bulk, completing on an
//    mbarrier), the A words of (i0..i0+RT-1, j) built by the CTA's threads from the
//    per-position loads table, whose global loads are issued one cut point ahead;
//  - all words are 32-bit and tagged: a finite value v is held as (v << tb) | tag, and
//    the maximum of two words with the same tag keeps the tag.  With rank tags (RT = 8)
//    the tag is the rank of (m, c') among the row block's admissible pairs in (m, c')
//    order, so the minimum over (m, c') of max(A, B) is one unsigned max and one min
//    per cell and pair and orders equal values as the packed key (v, j, m, c') does.
//    With width tags (RT = 4, for instances whose values need more bits) the tag is m:
//    the minimum over m orders (v, m), the next-link candidates c' are visited in
//    increasing order and one replaces the cut point's best only when strictly smaller.
//    Across cut points (visited in increasing j) a later one wins only with a strictly
//    smaller value, so each cell keeps its best word and its cut point (and c').
//  - a width whose stage fits no strategy at this position in any row of the block has
//    no finite A word and can only give no value: the A-word build records the widths
//    that have one (a mask per cut point), and the whole CTA skips the others, as the
//    recurrence itself skips transitions without a load.
// Values up to vmax = 2^(32 - tb) - 3 are exact.  A larger finite value saturates to
// vmax + 1: it can neither win nor tie against an exact value, so every cell whose
// optimum is at most vmax still gets its exact key, and a cell whose optimum is
// saturated flags its instance, which the 64-bit streaming variant then solves again
// (word mode 3; the later positions' launches skip a flagged instance).  Every
// launch writes the canonical tables (int64 values, uint32 arguments) that the
// backtrack and the tests read, and a 32-bit copy of its position for the next launch.
// Its bulk-copy waits are bounded: a wait that gives up marks the instance
// NEST_TIMED_OUT.
#include "nest_sweep.cuh"

namespace nest {

namespace {

constexpr int kLCols = 4;      // device counts per thread
constexpr int kLMaxThreads = 128;

// Shared-memory plan (byte offsets) and the strides of the layered kernels.
struct LayPlan {
    int NT;      // threads per CTA: one per 4 device counts, rounded up to warps
    int Dx;      // device counts per 32-bit row in global memory (d = 1 .. Dx)
    int XOFF;    // index of d = 0 in a shared row (= 3 mod 4, so that d = 1 starts 16 bytes in)
    int ROWW;    // words per shared row
    int Emax;    // (m, c') pairs per row block, at most
    int NIB;     // row blocks of 8 states per candidate (states 1 .. Nmax-1)
    int64_t mbar, X, rk, dec, fin, A, B, total;
};

__host__ __device__ inline LayPlan lay_plan(const Geo &g, int CT, int RT) {
    LayPlan s;
    s.NT = ((g.Dumax + kLCols - 1) / kLCols + 31) / 32 * 32;
    s.Dx = g.Dx;
    s.XOFF = (((1 << (g.Kmax - 1)) + 3) & ~3) + 3;
    s.ROWW = (s.XOFF + kLCols * s.NT + 1 + 3) & ~3;
    s.Emax = CT * g.Kmax;
    s.NIB = (g.Nmax - 1 + RT - 1) / RT;
    int64_t off = 0;
    s.mbar = off;
    off += 16;
    s.X = off;
    off = align_up(off + 8 * int64_t(g.Nmax + 1) * CT, 16);
    s.rk = off;                          // int32 [CT][16]
    off += 4 * 16 * CT;
    s.dec = off;                         // int32 [Emax]: (m << 4) | c'
    off = align_up(off + 4 * int64_t(s.Emax), 16);
    s.fin = off;                         // uint32 [3]: per cut point (in turn), the widths with a load
    off += 16;
    s.A = off;                           // uint32 [2][Emax][RT]
    off += 2 * 4 * int64_t(s.Emax) * RT;
    s.B = off;                           // uint32 [2][CT][ROWW]
    off += 2 * 4 * int64_t(CT) * s.ROWW;
    s.total = align_up(off, 128);
    return s;
}

// Row blocks per instance: the first stage (state 0, no input link), then RT-state
// blocks of states 1 .. Nmax-1 for each input candidate, the blocks with the most cut
// points first.
__host__ __device__ inline int lay_blocks(const Geo &g, int CT, int RT) { return 1 + lay_plan(g, CT, RT).NIB * CT; }

// Row (p, i, c) of the 32-bit copy of the DP values: d = 1 .. Dx at [d - 1].
__device__ __forceinline__ uint32_t *dp32_row(const PassArgs &a, int b, int p, int i, int c) {
    return reinterpret_cast<uint32_t *>(a.ws + a.w.dp32) +
           (((int64_t(b) * a.g.Pcap + (p - 1)) * a.g.Nmax + i) * a.g.Cmax + c) * a.g.Dx;
}

__device__ __forceinline__ int layers_of(const unsigned char *pb, const PassArgs &a, const PrepHdr *ph, int i) {
    if (!ph->graph) return ph->L - i;
    return __popcll(reinterpret_cast<const uint64_t *>(pb + a.pl.umask)[i]);
}

// Position 1: the last stage [i, L) alone, every cell (i, d, c) of every instance.
// One CTA per (instance, state i); 64-bit arithmetic (it also serves the instances that
// go on to the 64-bit streaming sweep); the 32-bit row is written for the others.
__global__ void __launch_bounds__(256) sweep_layer1_kernel(PassArgs a) {
    pdl_wait();
    pdl_trigger();
    const Geo &g = a.g;
    const int b = blockIdx.x / g.Nmax, i = blockIdx.x % g.Nmax;
    PrepHdr *ph = prep_hdr(a, b);
    if (ph->status != NEST_SOLVED) return;
    const int L = ph->L;
    if (i >= L) return;
    const LayWords w = lay_words(ph);
    const unsigned char *pb = reinterpret_cast<const unsigned char *>(ph);
    const int64_t *X = reinterpret_cast<const int64_t *>(pb + a.pl.X);
    const Inst s = load_inst(a, ph, b);
    const uint64_t *lrow = s.loads + (row_offset(i, L) + (L - i - 1)) * g.Kpad;   // position 1, pair (i, L)
    const int Dx = g.Dx;
    const int C = ph->C, K = ph->K, Du = ph->Du;
    bool sat = false;
    for (int e = threadIdx.x; e < C * (Dx + 1); e += blockDim.x) {
        const int c = e / (Dx + 1), d = e % (Dx + 1);
        uint64_t best = kInf;
        const bool cell = d >= 1 && d <= Du && (i > 0 || c == 0) && (i == 0 || ph->mlim[c] >= 0);
        if (cell) {
            const int ml = i == 0 ? K - 1 : (ph->mlim[c] < K - 1 ? ph->mlim[c] : K - 1);
            const int64_t xf = i > 0 ? X[int64_t(i) * g.Cmax + c] : 0;
            for (int m = 0; m <= ml && (1 << m) <= d; m++) {
                const uint64_t lw = lrow[m];
                if (lw == kInf) continue;
                const int64_t v = int64_t(lw >> 16) + xf;
                if (v >= kCap) continue;
                const uint64_t key = (uint64_t(v) << 24) | (uint64_t(L) << 8) | (uint64_t(m) << 4);
                best = key < best ? key : best;
            }
        }
        if (d <= Du) write_cell(s, g.Dpad, 1, i, c, d, best);
        if (w.ok && d >= 1) {
            const uint64_t v = best >> 24;
            sat |= best != kInf && v > w.vmax;
            dp32_row(a, b, 1, i, c)[d - 1] = best == kInf ? w.nmask : uint32_t(v > w.vmax ? w.vmax + 1 : v) << w.tb;
        }
    }
    if (__syncthreads_or(sat) && threadIdx.x == 0) atomicOr(&ph->lay_sat, 1);
}

// Position p >= 2 for every instance whose words take tag mode TW (0 rank, 1 width).
// blockIdx.x = instance * blocks + row block.
template <int CT, int RT, int TW>
__global__ void __launch_bounds__(kLMaxThreads) sweep_layer_kernel(PassArgs a, int p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Geo &g = a.g;
    const LayPlan lp = lay_plan(g, CT, RT);
    const int NB = 1 + lp.NIB * CT;
    const int b = blockIdx.x / NB, blk = blockIdx.x % NB;
    PrepHdr *ph = prep_hdr(a, b);
    // the instance's tag mode comes from the prep and stage-loads tables, which are
    // complete by now (every launch of this sweep waits for its predecessor before it
    // lets its own dependents start): the other mode's CTAs leave at once
    if (ph->status != NEST_SOLVED || p > ph->P || lay_words(ph).mode != TW) return;
    pdl_wait();
    pdl_trigger();
    const LayWords w = lay_words(ph);
    if (lay_leaves(ph)) return;   // the streaming sweep solves it (a flag the previous launch may set)
    const int L = ph->L, C = ph->C, K = ph->K, Du = ph->Du;
    const bool first = blk == 0;
    const int c = first ? 0 : (blk - 1) % CT;
    const int i0 = first ? 0 : 1 + ((blk - 1) / CT) * RT;
    if ((!first && c >= C) || i0 >= L) return;
    const unsigned char *pb = reinterpret_cast<const unsigned char *>(ph);
    const Inst s = load_inst(a, ph, b);
    const int tid = threadIdx.x, NT = lp.NT;

    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + lp.mbar);
    int64_t *Xs = reinterpret_cast<int64_t *>(smem + lp.X);   // [Nmax + 1][CT]
    int *rk = reinterpret_cast<int *>(smem + lp.rk);          // [CT][16] slot of (m, c') in A
    int *dec = reinterpret_cast<int *>(smem + lp.dec);        // [Emax]: (m << 4) | c'
    uint32_t *As = reinterpret_cast<uint32_t *>(smem + lp.A);
    uint32_t *Bs = reinterpret_cast<uint32_t *>(smem + lp.B);
    // per cut point, a mask of the widths m for which some row has a finite load; a width
    // with none relaxes nothing (max(no value, B) = no value).  Three words in turn: the
    // one built for cut point j + 1, the one read for j, and the one read for j - 1, which
    // is cleared while j is relaxed (no barrier separates a clear from the next build)
    uint32_t *fmw = reinterpret_cast<uint32_t *>(smem + lp.fin);

    // the widths a row block admits with each next-link candidate
    const int mlimc = first ? K - 1 : (ph->mlim[c] < K - 1 ? ph->mlim[c] : K - 1);
    int lim[CT];
#pragma unroll
    for (int c2 = 0; c2 < CT; c2++) {
        const int ml = c2 < C ? ph->mlim[c2] : -1;
        lim[c2] = ml < 0 || mlimc < 0 ? -1 : (ml < mlimc ? ml : mlimc);
    }
    // the states of the block, and whether each has a cell at position p
    bool act[RT];
#pragma unroll
    for (int r = 0; r < RT; r++) {
        const int i = i0 + r;
        act[r] = (first ? r == 0 : i < L) && p <= layers_of(pb, a, ph, i) && mlimc >= 0;
    }
    bool any = false;
#pragma unroll
    for (int r = 0; r < RT; r++) any |= act[r];
    const int jlo = i0 + 1;
    const int jhi = ph->graph ? L - 1 : (L - p + 1 < L - 1 ? L - p + 1 : L - 1);

    if (tid == 0) {
        int e = 0;
        for (int q = 0; q < 16 * CT; q++) rk[q] = -1;
        for (int m = 0; m < 16; m++)
            for (int c2 = 0; c2 < CT; c2++)
                if (m <= lim[c2]) {
                    rk[c2 * 16 + m] = e;
                    dec[e] = (m << 4) | c2;
                    e++;
                }
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        const int64_t *Xg = reinterpret_cast<const int64_t *>(pb + a.pl.X);
        for (int e = tid; e < (L + 1) * CT; e += NT) {
            const int q = e / CT, c2 = e % CT;
            Xs[e] = c2 < C ? Xg[int64_t(q) * g.Cmax + c2] : 0;
        }
        // every shared row starts as caps (no value); the copies fill d = 1 .. Dx
        for (int e = tid; e < 2 * CT * lp.ROWW; e += NT) Bs[e] = w.nmask;
        if (tid < 3) fmw[tid] = 0;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    const int64_t spin = a.spin_limit == 0 ? kDefaultSpin : a.spin_limit;
    const uint32_t row_bytes = uint32_t(4 * lp.Dx);
    const int warp = tid >> 5;
    // widest width any lane of this warp can use: 2^m <= d - (p - 1) for its largest d
    const int dmax_w = kLCols * (32 * warp + 32) < Du ? kLCols * (32 * warp + 32) : Du;
    int mwarp = -1;
    while (mwarp + 1 < K && (1 << (mwarp + 1)) <= dmax_w - (p - 1)) mwarp++;

    // A words of cut point j: thread q takes (r, m) = (q / K, q % K) for q = tid + k NT
    constexpr int kPre = (RT * 16 + 31) / 32;
    const int npair = RT * K;
    uint64_t pre[kPre];
    auto fetch = [&](int j) {
#pragma unroll
        for (int k = 0; k < kPre; k++) {
            const int q = tid + k * NT;
            pre[k] = kInf;
            if (q < npair) {
                const int r = q / K, m = q % K, i = i0 + r;
                if (act[r] && j > i && m <= mlimc)
                    pre[k] = s.loads[int64_t(p - 1) * s.pos_loads + (row_offset(i, L) + (j - i - 1)) * g.Kpad + m];
            }
        }
    };
    auto build = [&](int j, int buf, int slot) {   // every thread calls it
        uint32_t *Ab = As + buf * lp.Emax * RT;
        uint32_t bits = 0;   // widths with a finite load in one of this thread's rows
#pragma unroll
        for (int k = 0; k < kPre; k++) {
            const int q = tid + k * NT;
            if (q >= npair) continue;
            const int r = q / K, m = q % K, i = i0 + r;
            const int64_t base = pre[k] == kInf ? -1 : int64_t(pre[k] >> 16) + Xs[int64_t(i) * CT + c];
            bits |= base < 0 ? 0u : 1u << m;
#pragma unroll
            for (int c2 = 0; c2 < CT; c2++) {
                const int e = rk[c2 * 16 + m];
                if (e < 0) continue;
                const int64_t v = base + Xs[int64_t(j) * CT + c2];
                const uint32_t vv = v > int64_t(w.vmax) ? w.vmax + 1 : uint32_t(v);   // saturated
                Ab[e * RT + r] = base < 0 ? ~0u : (vv << w.tb) | uint32_t(TW ? m : e);
            }
        }
        bits = __reduce_or_sync(0xFFFFFFFFu, bits);
        if ((tid & 31) == 0 && bits) atomicOr(&fmw[slot], bits);
    };
    auto issue = [&](int j, int buf) {   // thread 0: the B rows (j, c') of position p - 1
        uint32_t bytes = 0;
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++) bytes += lim[c2] >= 0 ? row_bytes : 0u;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(&mbar[buf], bytes);
#pragma unroll
        for (int c2 = 0; c2 < CT; c2++)
            if (lim[c2] >= 0)
                bulk_g2s(Bs + (buf * CT + c2) * lp.ROWW + lp.XOFF + 1, dp32_row(a, b, p - 1, j, c2), row_bytes,
                         &mbar[buf]);
    };

    // the running best word and argument of each of the thread's RT x 4 cells (rank
    // tags: the cut point; width tags: (j << 4) | c')
    uint32_t rw[RT][kLCols], rj[RT][kLCols];
#pragma unroll
    for (int r = 0; r < RT; r++)
#pragma unroll
        for (int k = 0; k < kLCols; k++) {
            rw[r][k] = ~0u;
            rj[r][k] = 0;
        }
    uint32_t phase = 0, pending = 0;   // bit q: mbarrier q's parity, a copy on it in flight
    bool aborted = false;
    const int t = tid;   // columns d = 4t + 1 .. 4t + 4

    if (any && jlo <= jhi) {
        if (tid == 0) {
            issue(jlo, 0);
            pending = 1;
        }
        fetch(jlo);
        build(jlo, 0, 0);
        __syncthreads();
        int slot = 0;   // mask word of cut point j: (j - jlo) mod 3
        for (int j = jlo; j <= jhi; j++) {
            const int buf = (j - jlo) & 1;
            const int slot1 = slot == 2 ? 0 : slot + 1, slot2 = slot1 == 2 ? 0 : slot1 + 1;
            if (tid == 0) fmw[slot2] = 0;   // last read for cut point j - 1, next built for j + 2
            const bool more = j < jhi && !aborted;
            if (more) {
                if (tid == 0) {
                    issue(j + 1, buf ^ 1);
                    pending |= 1u << (buf ^ 1);
                }
                fetch(j + 1);
            }
            const bool ok = !aborted && mbar_wait(&mbar[buf], (phase >> buf) & 1, spin);
            if (ok) {
                phase ^= 1u << buf;
                pending &= ~(1u << buf);
                uint32_t cw[RT][kLCols];   // best over the pairs (m, c') of this cut point
                uint32_t jw[TW ? RT : 1][kLCols], jc[TW ? RT : 1][kLCols];
#pragma unroll
                for (int r = 0; r < RT; r++)
#pragma unroll
                    for (int k = 0; k < kLCols; k++) cw[r][k] = ~0u;
                if constexpr (TW) {
#pragma unroll
                    for (int r = 0; r < RT; r++)
#pragma unroll
                        for (int k = 0; k < kLCols; k++) {
                            jw[r][k] = ~0u;
                            jc[r][k] = 0;
                        }
                }
                const uint32_t *Ab = As + buf * lp.Emax * RT;
                // the widths with a finite load in some row at this cut point
                const uint32_t fmask = fmw[slot];
                auto relax = [&](uint4 B, int e, uint32_t tag) {
                    const uint32_t bb[4] = {B.x | tag, B.y | tag, B.z | tag, B.w | tag};
                    uint32_t aa[RT];
#pragma unroll
                    for (int h = 0; h < RT / 4; h++) {
                        const uint4 a4 = reinterpret_cast<const uint4 *>(Ab + e * RT)[h];
                        aa[4 * h] = a4.x;
                        aa[4 * h + 1] = a4.y;
                        aa[4 * h + 2] = a4.z;
                        aa[4 * h + 3] = a4.w;
                    }
#pragma unroll
                    for (int r = 0; r < RT; r++)
#pragma unroll
                        for (int k = 0; k < kLCols; k++) cw[r][k] = min(cw[r][k], max(aa[r], bb[k]));
                };
                // a cut point whose stages fit no strategy at this position gives nothing
                if (fmask != 0) {
#pragma unroll
                for (int c2 = 0; c2 < CT; c2++) {
                    const int mm = lim[c2] < mwarp ? lim[c2] : mwarp;
                    if (mm < 0) continue;
                    const uint32_t *row = Bs + (buf * CT + c2) * lp.ROWW + lp.XOFF + 1;   // row[x - 1] = B[x]
                    const int *rkc = rk + c2 * 16;
                    const uint4 U0 = *reinterpret_cast<const uint4 *>(row + 4 * t);       // B[4t+1 .. 4t+4]
                    const uint4 U1 = *reinterpret_cast<const uint4 *>(row + 4 * t - 4);   // B[4t-3 .. 4t]
                    if (fmask & 1) relax(make_uint4(U1.w, U0.x, U0.y, U0.z), rkc[0], TW ? 0u : uint32_t(rkc[0]));   // 2^0
                    if (mm >= 1 && (fmask & 2))
                        relax(make_uint4(U1.z, U1.w, U0.x, U0.y), rkc[1], TW ? 1u : uint32_t(rkc[1]));
                    if (mm >= 2 && (fmask & 4)) relax(U1, rkc[2], TW ? 2u : uint32_t(rkc[2]));   // 2^2
                    for (int m = 3; m <= mm; m++)
                        if ((fmask >> m) & 1)
                            relax(*reinterpret_cast<const uint4 *>(row + 4 * t - (1 << m)), rkc[m],
                                  TW ? uint32_t(m) : uint32_t(rkc[m]));
                    if constexpr (TW) {
                        // this candidate's best (v, m) replaces the cut point's only when
                        // strictly smaller: equal ones keep the smaller c'
#pragma unroll
                        for (int r = 0; r < RT; r++)
#pragma unroll
                            for (int k = 0; k < kLCols; k++) {
                                const bool take = cw[r][k] < jw[r][k];
                                jw[r][k] = take ? cw[r][k] : jw[r][k];
                                jc[r][k] = take ? uint32_t(c2) : jc[r][k];
                                cw[r][k] = ~0u;
                            }
                    }
                }
                // a later cut point wins only with a strictly smaller value
#pragma unroll
                for (int r = 0; r < RT; r++)
#pragma unroll
                    for (int k = 0; k < kLCols; k++) {
                        const uint32_t cand = TW ? jw[TW ? r : 0][k] : cw[r][k];
                        const bool take = cand < (rw[r][k] & w.nmask);
                        rw[r][k] = take ? cand : rw[r][k];
                        rj[r][k] = take ? (TW ? uint32_t(j) << 4 | jc[TW ? r : 0][k] : uint32_t(j)) : rj[r][k];
                    }
                }
            }
            if (more) build(j + 1, buf ^ 1, slot1);
            aborted = __syncthreads_or(!ok) != 0;
            slot = slot1;
        }
    }

    // the cells: canonical tables and the 32-bit row for position p + 1
    bool sat = false;
#pragma unroll
    for (int r = 0; r < RT; r++) {
        const int i = i0 + r;
        if (first ? r != 0 : i >= L) continue;
        uint32_t wd[kLCols];
#pragma unroll
        for (int k = 0; k < kLCols; k++) {
            const int d = kLCols * t + 1 + k;
            const uint32_t v = rw[r][k] >> w.tb;
            const bool fin = v <= w.vmax;
            sat |= v == w.vmax + 1 && d <= Du;
            wd[k] = fin && d <= Du ? (rw[r][k] & w.nmask) : w.nmask;
            if (d <= Du) {
                const uint32_t tag = rw[r][k] & ~w.nmask;
                // (j << 8) | (m << 4) | c'
                const uint32_t arg = TW ? (rj[r][k] >> 4) << 8 | tag << 4 | (rj[r][k] & 15)
                                        : rj[r][k] << 8 | uint32_t(dec[tag]);
                const uint64_t key = fin ? (uint64_t(v) << 24) | uint64_t(arg) : kInf;
                write_cell(s, g.Dpad, p, i, c, d, key);
            }
        }
        if (kLCols * t < lp.Dx)
            *reinterpret_cast<uint4 *>(dp32_row(a, b, p, i, c) + kLCols * t) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        if (tid == 0) write_cell(s, g.Dpad, p, i, c, 0, kInf);
    }
    // state 0 has no input link: its cells of the other candidates have no value
    if (first)
        for (int e = tid; e < (C - 1) * (Du + 1); e += NT) write_cell(s, g.Dpad, p, 0, 1 + e / (Du + 1), e % (Du + 1), kInf);
    if (__syncthreads_or(sat) && tid == 0) atomicOr(&ph->lay_sat, 1);
    if (tid == 0) {
        // drain copies still in flight (only after a wait gave up)
        for (int q = 0; q < 2; q++)
            if ((pending >> q) & 1) mbar_wait(&mbar[q], (phase >> q) & 1, kDefaultSpin);
        if (aborted) ph->status = NEST_TIMED_OUT;
    }
}

template <int CT, int RT, int TW>
int launch_layer_mode(const PassArgs &a, void *stream, int p) {
    const LayPlan lp = lay_plan(a.g, CT, RT);
    const size_t smem = size_t(lp.total);
    if (int rc = cuda_status(cudaFuncSetAttribute(sweep_layer_kernel<CT, RT, TW>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                             "layered sweep smem attribute"))
        return rc;
    const dim3 grid(unsigned(int64_t(a.n) * lay_blocks(a.g, CT, RT)));
    return launch_kernel(sweep_layer_kernel<CT, RT, TW>, grid, dim3(unsigned(lp.NT)), smem, stream, 1,
                         "layered sweep launch", a, p);
}

// Position p: the rank-tag launch (8 states per thread), then the width-tag launch (4
// states per thread); each leaves the other's instances alone.
template <int CT>
int launch_layer_ct(const PassArgs &a, void *stream, int p) {
    if (int rc = launch_layer_mode<CT, 8, 0>(a, stream, p)) return rc;
    return launch_layer_mode<CT, 4, 1>(a, stream, p);
}

}  // namespace

int64_t layered_smem_bytes(const Geo &g) { return lay_plan(g, ct_of(g.Cmax), 8).total; }

int launch_layered(const PassArgs &a, void *stream) {
    const Geo &g = a.g;
    if (int rc = launch_kernel(sweep_layer1_kernel, dim3(unsigned(int64_t(a.n) * g.Nmax)), dim3(256), 0, stream, 1,
                               "layered sweep (position 1) launch", a))
        return rc;
    const int CT = ct_of(g.Cmax);
    for (int p = 2; p <= g.Pcap; p++) {
        int rc = CT == 1 ? launch_layer_ct<1>(a, stream, p)
                 : CT == 2 ? launch_layer_ct<2>(a, stream, p)
                 : CT == 3 ? launch_layer_ct<3>(a, stream, p)
                           : launch_layer_ct<4>(a, stream, p);
        if (rc) return rc;
    }
    return NEST_OK;
}

}  // namespace nest
