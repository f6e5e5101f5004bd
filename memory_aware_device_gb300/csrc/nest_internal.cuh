// Internal layouts and helpers of the GB300 placement-DP solver.
//
// Method: "Nest: Network- and Memory-Aware Device Placement for Distributed Deep
// Learning" (Nest), §3.3 memory model, §4 Eq. 3 and load(), Appendix K Algorithm 1.
// The public ABI is include/nest.h; everything here is private to the library.
#pragma once

#include <cstdint>

#include "../../include/nest.h"
#include "nest_divide.cuh"

namespace nest {

constexpr int64_t kCap = (int64_t(1) << 40) - 1;   // stage times >= kCap are infeasible
constexpr uint64_t kInf = ~uint64_t(0);             // "no value" word / key
constexpr uint32_t kNoArg = 0xFFFFFFu;              // argument field of an empty DP cell
constexpr int kLogL = 8;                            // sparse-table levels: 2^8 > 255 layers
constexpr int kMaxStates = 256;                     // DP states per instance (8-bit state index)

__host__ __device__ inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Batch geometry derived from nest_dims.
struct Geo {
    int32_t B, Lmax, Tmax, Cmax, Smax, Pcap, Dumax, Vmax;
    int32_t Nmax;  // last DP state index of any instance: max(Lmax, Vmax)
    int32_t NP;    // pairs of states (i, j), 0 <= i < j <= Nmax
    int32_t Kmax;  // widths unit * 2^m, m < Kmax
    int32_t Kpad;  // Kmax rounded up to even (16-byte rows)
    int32_t Spad;  // Smax rounded up to even
    int32_t Dpad;  // Dumax + 1 rounded up to a multiple of 4 (rows of 16-byte multiples)
    int32_t Dx;    // Dumax rounded up to a multiple of 4 (32-bit rows of device counts 1 .. Dx)
    int32_t pad_;
};

inline bool make_geo(const nest_dims &d, Geo &g) {
    if (d.B < 0 || d.Lmax < 1 || d.Lmax > 255 || d.Tmax < 1 || d.Tmax > 8 || d.Cmax < 1 ||
        d.Cmax > 15 || d.Smax < 1 || d.Smax > 4095 || d.Pcap < 1 || d.Pcap > 31 || d.Dumax < 1 ||
        d.Dumax > 512 || d.Vmax < 0 || d.Vmax >= kMaxStates)
        return false;
    g.B = d.B;
    g.Lmax = d.Lmax;
    g.Tmax = d.Tmax;
    g.Cmax = d.Cmax;
    g.Smax = d.Smax;
    g.Pcap = d.Pcap;
    g.Dumax = d.Dumax;
    g.Vmax = d.Vmax;
    g.Nmax = d.Lmax > d.Vmax ? d.Lmax : d.Vmax;
    g.NP = g.Nmax * (g.Nmax + 1) / 2;
    int K = 0;
    while ((1 << K) <= d.Dumax) K++;
    g.Kmax = K;
    g.Kpad = (K + 1) & ~1;
    g.Spad = (d.Smax + 1) & ~1;
    g.Dpad = (d.Dumax + 4) & ~3;
    g.Dx = (d.Dumax + 3) & ~3;
    g.pad_ = 0;
    return true;
}

// Offsets inside one instance record (public layout, see nest.h).
inline void record_layout(const Geo &g, nest_layout &o) {
    int64_t off = align_up(sizeof(nest_record_header), 16);
    auto take = [&](int64_t bytes) {
        int64_t at = off;
        off = align_up(off + bytes, 16);
        return at;
    };
    o.fl = take(8 * g.Lmax);
    o.pd = take(8 * g.Lmax);
    o.pe = take(8 * g.Lmax);
    o.ao = take(8 * g.Lmax);
    o.aw = take(8 * g.Lmax);
    o.a2a = take(8 * g.Lmax);
    o.moe = take(g.Lmax);
    o.G = take(8 * g.Tmax);
    o.bw = take(8 * g.Tmax);
    o.lat = take(8 * g.Tmax);
    o.cand = take(4 * g.Cmax);
    o.strat = take(16 * g.Smax);
    o.succ = take(8 * g.Lmax);
    o.record_bytes = align_up(off, 256);
}

// Per-instance preparation record written by the prep kernel.
struct PrepHdr {
    int32_t status;  // NEST_SOLVED (0) when the instance is valid, NEST_BAD_INPUT otherwise;
                     // the sweep raises it to NEST_TIMED_OUT when a wait gives up
    int32_t L;       // last DP state: the empty set (layers of a chain, up-sets - 1 of a graph)
    int32_t D, unit, lu, Du, K, T, C, S, P;
    uint32_t maxX32;     // largest link cost X, saturated at 2^31 - 1 (prep)
    uint32_t maxload32;  // largest finite per-position load tau*, saturated (reduction)
    int32_t schedule;    // 0 = 1F1B, 1 = GPipe
    int32_t graph;       // 0 = chain, 1 = states are the up-sets of a layer DAG
    int32_t layers;      // layers of the instance
    int32_t lay_sat;     // the layered sweep met a value beyond its 32-bit words (the
                         // streaming sweep then solves the instance again)
    int32_t ngrp;        // strategy groups: runs of equal (t, cp, e) in the sorted strategy list
    int32_t ngd;         // dense groups: runs of equal (t, cp), each a run of strategy groups
    int32_t lay_pad;
    int64_t R, M, budget, opt;
    int64_t G[8], bw[8], lat[8];
    int32_t cand[16];
    int32_t mlim[16];    // largest m with 2 * unit * 2^m <= G[cand c], -1 if none
    int8_t tier_log[16]; // smallest tier whose groups hold 2^x devices, x = 0 .. 13
    Divisor bwdiv[8];    // invariant divisors for bw[t]
    Divisor Mdiv, Rdiv;  // and for M and R
};
static_assert(sizeof(PrepHdr) % 16 == 0, "PrepHdr alignment");

enum { kFl = 0, kPd, kPe, kAo, kAw, kA2, kNm, kNumPfx };

struct PrepLayout {
    int64_t pfx;    // int64 [kNumPfx][Lmax + 1] prefix sums over layers
    int64_t ain;    // int64 [Nmax + 1] bytes entering each state (link volume, stashed input)
    int64_t umask;  // uint64 [Nmax + 1] layers of each state (chains of <= 64 layers, graphs)
    int64_t awst;   // int64 [kLogL][Lmax] sparse table of max(aw)
    int64_t X;      // int64 [Nmax + 1][Cmax] link cost into each state per candidate
    int64_t strat;  // uint32 [Smax] packed log2 t | log2 cp << 4 | log2 e << 8 | z << 12 | r << 14
    int64_t ssort;  // uint32 [Smax] the codes sorted by (t, cp, e, z, r, s), each | s << 16
    int64_t sgrp;   // uint32 [Smax + 1] start of each strategy group in ssort (ngrp + 1 entries)
    int64_t sgd;    // uint32 [Smax + 1] first strategy group of each dense group (ngd + 1 entries)
    int64_t bytes;
};

__host__ __device__ inline PrepLayout prep_layout(const Geo &g) {
    PrepLayout p;
    int64_t off = sizeof(PrepHdr);
    p.pfx = off;
    off += 8 * int64_t(kNumPfx) * (g.Lmax + 1);
    p.ain = off;
    off += 8 * int64_t(g.Nmax + 1);
    p.umask = off;
    off += 8 * int64_t(g.Nmax + 1);
    p.awst = off;
    off += 8 * int64_t(kLogL) * g.Lmax;
    p.X = off;
    off += 8 * int64_t(g.Nmax + 1) * g.Cmax;
    p.strat = off;
    off += 4 * int64_t(g.Smax);
    p.ssort = off;
    off += 4 * int64_t(g.Smax);
    p.sgrp = off;
    off += 4 * int64_t(g.Smax + 1);
    p.sgd = off;
    off += 4 * int64_t(g.Smax + 1);
    p.bytes = align_up(off, 256);
    return p;
}

// Workspace regions for passes of `ch` instances.
struct WsLayout {
    int64_t prep, loads, dpv, dpa, dp32, total, cost, total_costs;
    int64_t prep_stride, cost_stride, loads_stride, dp_stride, dp32_stride;  // per instance (elements for tables)
};

__host__ __device__ inline WsLayout ws_layout(const Geo &g, int64_t ch) {
    WsLayout w;
    PrepLayout p = prep_layout(g);
    w.prep_stride = p.bytes;
    w.cost_stride = int64_t(g.NP) * g.Kmax * g.Spad;            // uint64 words
    w.loads_stride = int64_t(g.Pcap) * g.NP * g.Kpad;           // uint64 words
    w.dp_stride = int64_t(g.Pcap) * g.Nmax * g.Cmax * g.Dpad;   // cells
    w.dp32_stride = int64_t(g.Pcap) * g.Nmax * g.Cmax * g.Dx;   // 32-bit words (layered sweep)
    int64_t off = 0;
    w.prep = off;
    off = align_up(off + ch * w.prep_stride, 256);
    w.loads = off;
    off = align_up(off + ch * w.loads_stride * 8, 256);
    w.dpv = off;
    off = align_up(off + ch * w.dp_stride * 8, 256);
    w.dpa = off;
    off = align_up(off + ch * w.dp_stride * 4, 256);
    w.dp32 = off;
    off = align_up(off + ch * w.dp32_stride * 4, 256);
    w.total = off;
    w.cost = off;   // only with NEST_KEEP_COSTS
    off = align_up(off + ch * w.cost_stride * 8, 256);
    w.total_costs = off;
    return w;
}

__host__ __device__ inline int64_t plan_bytes(const Geo &g) {
    return align_up(int64_t(sizeof(nest_plan_header)) + int64_t(sizeof(nest_stage)) * g.Pcap, 8);
}

// Row offset of pair (i, i+1) among the pairs of states 0 .. L.
__host__ __device__ inline int64_t row_offset(int i, int L) {
    return int64_t(i) * L - int64_t(i) * (i - 1) / 2;
}

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Arguments shared by the kernels of one pass.
struct PassArgs {
    Geo g;
    WsLayout w;
    PrepLayout pl;
    nest_layout rl;
    const unsigned char *records;  // device, first instance of the pass
    unsigned char *ws;             // device workspace base
    int64_t *costs_out;            // device, first instance of the pass
    unsigned char *plans_out;      // device, first plan of the pass
    int64_t plan_stride;
    int32_t n;                     // instances in this pass
    int32_t cluster;               // sweep CTAs per instance
    int32_t jsplit;                // sweep threads per DP cell
    int32_t jc;                    // sweep j-chunk (layers staged per tile)
    int32_t threads;               // sweep threads per CTA
    int32_t resident;              // sweep variant: 1 = dp rows resident in shared memory
    int64_t spin_limit;            // polls per bounded wait (negative: give up at once)
    int32_t keep_costs;            // also write the stage-cost tensor
    int32_t word_mode;             // sweep launch takes: 0 every instance, 1 those on 32-bit
                                   // words only, 2 those on 64-bit words only, 3 (streaming)
                                   // those the layered sweep leaves (values beyond its words)
    int32_t fuse_walk;             // resident sweep: rank 0 of each cluster also writes the plan
                                   // (the final reduction and backtrack), no backtrack launch
    int32_t pad;
};

__host__ __device__ inline PrepHdr *prep_hdr(const PassArgs &a, int b) {
    return reinterpret_cast<PrepHdr *>(a.ws + a.w.prep + int64_t(b) * a.w.prep_stride);
}

// Maps a CUDA runtime status to NEST_OK / NEST_E_CUDA; with NEST_DEBUG set in the
// environment a failure is also reported on stderr with the call that failed.
int cuda_status(int err, const char *what);

// Programmatic dependent launch.  Every kernel of a pass is launched with
// programmatic stream serialization allowed, so it can be scheduled while the
// previous kernel on the stream is still running: it lets its own dependents launch
// at once (pdl_trigger) and waits for the previous kernel to complete and its memory
// to be visible (pdl_wait) before touching anything that kernel wrote.  Both are
// no-ops for a launch without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `fn(args...)` with the PDL attribute, plus a cluster shape when cluster > 1.
template <typename... KArgs, typename... Args>
int launch_kernel(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem, void *stream, int cluster,
                  const char *what, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = unsigned(cluster);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        na++;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cuda_status(cudaLaunchKernelEx(&cfg, fn, args...), what);
}

// Launchers (one translation unit each).
int launch_prep(const PassArgs &a, void *stream);
int launch_loads(const PassArgs &a, void *stream);
int launch_sweep(const PassArgs &a, void *stream);
int launch_backtrack(const PassArgs &a, void *stream);
// The layered sweep (nest_layered.cu): position 1, then one launch per position 2 .. Pcap.
int launch_layered(const PassArgs &a, void *stream);
int64_t layered_smem_bytes(const Geo &g);
// Dynamic shared memory of the streaming and resident sweep variants.
int64_t sweep_smem_bytes(const Geo &g, int jc, int jsplit, int threads);
int64_t sweep_resident_smem_bytes(const Geo &g, int cluster, int jsplit, int threads, int mode);

// Launch shape of the DP sweep for passes of n instances.  cluster_opt / jsplit_opt
// (0 = choose) and variant (0 = choose, 1 = resident, 2 = streaming, 3 = layered) come from
// nest_options.  With split set, the sweep is two launches: the resident shape above
// sized for the instances on 32-bit words alone (word_mode 1), then `wide` for those
// on 64-bit words (word_mode 2).  Returns NEST_OK, NEST_E_INVALID or NEST_E_LIMITS.
struct SweepShape {
    int cluster, jsplit, jc, threads, resident, resident_waves;
};
struct SweepConfig {
    int cluster, jsplit, jc, threads, resident, resident_waves;
    int split;
    SweepShape wide;
    int layered;   // 1: the layered sweep, then the streaming shape above for the instances it leaves
};
int sweep_configure(const Geo &g, int n, int cluster_opt, int jsplit_opt, int variant, SweepConfig &out);

}  // namespace nest
