// Backtrack: the final batch-time loop and the stage reconstruction of Nest
// (Network- and Memory-Aware Device Placement) Appendix K Algorithm 1.
//
// t_batch = min over stage counts p of v(dp[0][Du][p]) * (M + p - 1) (ties to the
// smaller p), then the plan is read back by following the argument field of each
// DP cell: (j, m, c') gives the end of the stage, its width unit * 2^m and the
// candidate of its outgoing link; the stage's strategy is the argument of the
// per-position strategy minimum.  Lanes of a warp evaluate the stage counts in
// parallel and a shuffle reduction picks the best (t, p); lane 0 then walks the plan.
#include <cuda_runtime.h>

#include "nest_internal.cuh"

namespace nest {

namespace {

__global__ void __launch_bounds__(128) backtrack_kernel(PassArgs a) {
    __shared__ int walk[4][32][2];   // per warp: stage q -> (i | j << 8 | m << 16 | c' << 20, p)
    pdl_wait();
    pdl_trigger();
    const int b = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31, wq = threadIdx.x >> 5;
    if (b >= a.n) return;   // whole warps
    const PrepHdr *ph = prep_hdr(a, b);
    nest_plan_header *hdr = reinterpret_cast<nest_plan_header *>(a.plans_out + int64_t(b) * a.plan_stride);
    nest_stage *st = reinterpret_cast<nest_stage *>(hdr + 1);
    int status = ph->status;
    const Geo &g = a.g;
    const int64_t row_cells = int64_t(g.Cmax) * g.Dpad;
    const int64_t pos_cells = int64_t(g.Lmax) * row_cells;
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
            walk[wq][n][0] = i | j << 8 | m << 16 | c2 << 20;
            walk[wq][n][1] = p;
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
        const int w = walk[wq][lane][0], p = walk[wq][lane][1];
        const int i = w & 0xFF, j = (w >> 8) & 0xFF, m = (w >> 16) & 0xF, c2 = (w >> 20) & 0xF;
        const uint64_t lw = loads[int64_t(p - 1) * g.NP * g.Kpad + (row_offset(i, L) + (j - i - 1)) * g.Kpad + m];
        st[lane].i = int16_t(i);
        st[lane].j = int16_t(j);
        st[lane].s = int16_t(lw & 0xFFFF);
        st[lane].c_next = int8_t(j < L ? c2 : -1);
        st[lane].reserved = 0;
        st[lane].k = ph->unit << m;
    }
    if (lane == 0) {
        hdr->status = NEST_SOLVED;
        hdr->n_stages = n;
        hdr->t_batch = bt;
        hdr->bottleneck = dpv[int64_t(bp - 1) * pos_cells + ph->Du];
        a.costs_out[b] = bt;
    }
}

}  // namespace

int launch_backtrack(const PassArgs &a, void *stream) {
    const int threads = 128;
    const int64_t total = int64_t(a.n) * 32;
    return launch_kernel(backtrack_kernel, dim3(unsigned((total + threads - 1) / threads)), dim3(threads), 0, stream, 1,
                         "backtrack launch", a);
}

}  // namespace nest
