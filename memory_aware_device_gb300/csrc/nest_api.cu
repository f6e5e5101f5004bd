// C ABI of the placement-DP solver (declared in include/nest.h).
//
// A call validates the batch dimensions on the host, then, for each chunk of
// instances, enqueues on the caller's stream: prep (validation, prefix sums, DP
// states, link costs), stage loads (cost build and strategy reduction), the DP sweep
// (two launches when split by word width) and, after a streaming sweep only, the
// backtrack (a resident sweep's clusters write their plans).  Nothing is allocated
// and no state survives the call.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "nest_internal.cuh"

namespace nest {

int cuda_status(int err, const char *what) {
    if (err == cudaSuccess) return NEST_OK;
    if (std::getenv("NEST_DEBUG"))
        std::fprintf(stderr, "nest: %s failed: %s\n", what, cudaGetErrorString(cudaError_t(err)));
    return NEST_E_CUDA;
}

}  // namespace nest

using namespace nest;

namespace {

// Instances per pass: the whole batch by default, at most 65535 (the stage-loads
// kernel indexes instances with blockIdx.y).
int32_t chunk_of(const nest_dims *dims, int32_t chunk) {
    if (chunk <= 0 || chunk > dims->B) chunk = dims->B;
    return chunk < 65535 ? chunk : 65535;
}

}  // namespace

extern "C" {

int nest_record_layout(const nest_dims *dims, nest_layout *out) {
    Geo g;
    if (!dims || !out) return NEST_E_INVALID;
    if (!make_geo(*dims, g)) return NEST_E_LIMITS;
    record_layout(g, *out);
    return NEST_OK;
}

size_t nest_plan_bytes(const nest_dims *dims) {
    Geo g;
    if (!dims || !make_geo(*dims, g)) return 0;
    return size_t(plan_bytes(g));
}

size_t nest_workspace_size(const nest_dims *dims, int32_t chunk) {
    Geo g;
    if (!dims || !make_geo(*dims, g)) return 0;
    const int32_t ch = chunk_of(dims, chunk);
    return size_t(ws_layout(g, ch < 1 ? 1 : ch).total);
}

size_t nest_workspace_size_costs(const nest_dims *dims, int32_t chunk) {
    Geo g;
    if (!dims || !make_geo(*dims, g)) return 0;
    const int32_t ch = chunk_of(dims, chunk);
    return size_t(ws_layout(g, ch < 1 ? 1 : ch).total_costs);
}

int nest_workspace_layout(const nest_dims *dims, int32_t chunk, nest_ws_layout *out) {
    Geo g;
    if (!dims || !out) return NEST_E_INVALID;
    if (!make_geo(*dims, g)) return NEST_E_LIMITS;
    const int32_t ch = chunk_of(dims, chunk);
    const WsLayout w = ws_layout(g, ch < 1 ? 1 : ch);
    out->loads = w.loads;
    out->dpv = w.dpv;
    out->dpa = w.dpa;
    out->cost = w.cost;
    out->total = w.total;
    out->total_costs = w.total_costs;
    out->NP = g.NP;
    out->Kmax = g.Kmax;
    out->Kpad = g.Kpad;
    out->Spad = g.Spad;
    out->Dpad = g.Dpad;
    out->chunk = ch;
    out->N = g.Nmax;
    out->reserved = 0;
    return NEST_OK;
}

int nest_describe_launch(const nest_dims *dims, const nest_options *opt, nest_launch_desc *out) {
    if (!dims || !out) return NEST_E_INVALID;
    Geo g;
    if (dims->B < 0) return NEST_E_INVALID;
    if (!make_geo(*dims, g)) return NEST_E_LIMITS;
    const int32_t chunk = chunk_of(dims, opt ? opt->chunk : 0);
    SweepConfig cfg;
    const int rc = sweep_configure(g, chunk < 1 ? 1 : chunk, opt ? opt->sweep_cluster : 0,
                                   opt ? opt->sweep_jsplit : 0, opt ? opt->sweep_variant : 0, cfg);
    if (rc != NEST_OK) return rc;
    std::memset(out, 0, sizeof *out);
    out->chunks = dims->B == 0 ? 0 : (dims->B + chunk - 1) / chunk;
    // prep, stage loads, the sweep (two launches when split), and the backtrack unless
    // every sweep launch is resident (their clusters write the plans)
    const bool fuse = cfg.resident && (!cfg.split || cfg.wide.resident);
    // the layered sweep: position 1, two launches (rank and width tags) per later
    // position, the streaming launch for the instances beyond its words
    const int sweep_launches = cfg.layered ? 1 + 2 * (g.Pcap - 1) + 1 : 1 + (cfg.split ? 1 : 0);
    out->kernels_per_chunk = 2 + sweep_launches + (fuse ? 0 : 1);
    out->sweep_variant = cfg.layered ? 3 : cfg.resident ? 1 : 2;
    out->sweep_cluster = cfg.cluster;
    out->sweep_jsplit = cfg.jsplit;
    out->sweep_threads = cfg.threads;
    out->sweep_split = cfg.split;
    if (cfg.split) {
        out->wide_variant = cfg.wide.resident ? 1 : 2;
        out->wide_cluster = cfg.wide.cluster;
        out->wide_jsplit = cfg.wide.jsplit;
        out->wide_threads = cfg.wide.threads;
    }
    return NEST_OK;
}

// The DP sweep of one pass: one launch, or the 32-bit-word launch followed by the
// 64-bit-word one (each leaves the other's instances alone).
static int sweep_pass(PassArgs a, const SweepConfig &cfg, void *stream) {
    if (cfg.layered) {
        // the layered launches, then the streaming variant for the instances whose values
        // do not fit their words (its CTAs for the others exit at once)
        if (int rc = launch_layered(a, stream)) return rc;
        a.word_mode = 3;
        return launch_sweep(a, stream);
    }
    if (!cfg.split) {
        a.word_mode = 0;
        return launch_sweep(a, stream);
    }
    a.word_mode = 1;
    if (int rc = launch_sweep(a, stream)) return rc;
    a.word_mode = 2;
    a.cluster = cfg.wide.cluster;
    a.jsplit = cfg.wide.jsplit;
    a.jc = cfg.wide.jc;
    a.threads = cfg.wide.threads;
    a.resident = cfg.wide.resident;
    return launch_sweep(a, stream);
}

int nest_solve(const nest_dims *dims, const void *records, int64_t *costs_out, void *plans_out,
               void *workspace, size_t ws_bytes, void *stream, const nest_options *opt) {
    if (!dims) return NEST_E_INVALID;
    Geo g;
    if (dims->B < 0) return NEST_E_INVALID;
    if (!make_geo(*dims, g)) return NEST_E_LIMITS;
    if (dims->B == 0) return NEST_OK;
    if (!records || !costs_out || !plans_out || !workspace) return NEST_E_INVALID;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 || reinterpret_cast<uintptr_t>(records) % 256)
        return NEST_E_WORKSPACE;
    const int32_t chunk = chunk_of(dims, opt ? opt->chunk : 0);
    const WsLayout w = ws_layout(g, chunk);
    const uint32_t flags = opt ? opt->flags : 0u;
    if (flags & ~NEST_KEEP_COSTS) return NEST_E_INVALID;
    const bool keep = (flags & NEST_KEEP_COSTS) != 0;
    if (ws_bytes < size_t(keep ? w.total_costs : w.total)) return NEST_E_WORKSPACE;
    SweepConfig cfg;
    int rc = sweep_configure(g, chunk, opt ? opt->sweep_cluster : 0, opt ? opt->sweep_jsplit : 0,
                             opt ? opt->sweep_variant : 0, cfg);
    if (rc != NEST_OK) return rc;

    PassArgs a;
    std::memset(&a, 0, sizeof a);
    a.g = g;
    a.w = w;
    a.pl = prep_layout(g);
    record_layout(g, a.rl);
    a.ws = static_cast<unsigned char *>(workspace);
    a.plan_stride = plan_bytes(g);
    a.cluster = cfg.cluster;
    a.jsplit = cfg.jsplit;
    a.jc = cfg.jc;
    a.threads = cfg.threads;
    a.resident = cfg.resident;
    a.spin_limit = opt ? opt->spin_limit : 0;
    a.keep_costs = keep ? 1 : 0;
    a.fuse_walk = cfg.resident && (!cfg.split || cfg.wide.resident) ? 1 : 0;
    cudaEvent_t *ev = opt ? reinterpret_cast<cudaEvent_t *>(opt->events) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto mark = [&](int chunk_idx, int k) {
        return ev && ev[5 * chunk_idx + k] ? cuda_status(cudaEventRecord(ev[5 * chunk_idx + k], st), "cudaEventRecord")
                                           : NEST_OK;
    };
    int ci = 0;
    for (int32_t first = 0; first < dims->B; first += chunk, ci++) {
        a.n = dims->B - first < chunk ? dims->B - first : chunk;
        a.records = static_cast<const unsigned char *>(records) + int64_t(first) * a.rl.record_bytes;
        a.costs_out = costs_out + first;
        a.plans_out = static_cast<unsigned char *>(plans_out) + int64_t(first) * a.plan_stride;
        if ((rc = mark(ci, 0)) || (rc = launch_prep(a, st)) || (rc = mark(ci, 1)) || (rc = launch_loads(a, st)) ||
            (rc = mark(ci, 2)) || (rc = sweep_pass(a, cfg, st)) || (rc = mark(ci, 3)) ||
            (!a.fuse_walk && (rc = launch_backtrack(a, st))) || (rc = mark(ci, 4)))
            return rc;
    }
    return NEST_OK;
}

size_t nest_workspace_size_host(const nest_dims *dims, int32_t chunk) {
    Geo g;
    if (!dims || !make_geo(*dims, g)) return 0;
    nest_layout rl;
    record_layout(g, rl);
    const int64_t B = dims->B;
    return size_t(align_up(B * rl.record_bytes, 256) + align_up(8 * B, 256) + align_up(B * plan_bytes(g), 256) +
                  int64_t(nest_workspace_size(dims, chunk)));
}

int nest_solve_host(const nest_dims *dims, const void *records_host, int64_t *costs_host, void *plans_host,
                    void *workspace, size_t ws_bytes, void *stream, const nest_options *opt) {
    if (!dims) return NEST_E_INVALID;
    Geo g;
    if (dims->B < 0) return NEST_E_INVALID;
    if (!make_geo(*dims, g)) return NEST_E_LIMITS;
    if (dims->B == 0) return NEST_OK;
    if (!records_host || !costs_host || !plans_host || !workspace) return NEST_E_INVALID;
    if (opt && opt->flags) return NEST_E_INVALID;   // the host entry keeps no intermediate tables
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return NEST_E_WORKSPACE;
    if (ws_bytes < nest_workspace_size_host(dims, opt ? opt->chunk : 0)) return NEST_E_WORKSPACE;
    nest_layout rl;
    record_layout(g, rl);
    const int64_t B = dims->B;
    unsigned char *base = static_cast<unsigned char *>(workspace);
    unsigned char *rec_d = base;
    int64_t *costs_d = reinterpret_cast<int64_t *>(base + align_up(B * rl.record_bytes, 256));
    unsigned char *plans_d = reinterpret_cast<unsigned char *>(costs_d) + align_up(8 * B, 256);
    unsigned char *ws = plans_d + align_up(B * plan_bytes(g), 256);
    const size_t ws_left = ws_bytes - size_t(ws - base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = cuda_status(
        cudaMemcpyAsync(rec_d, records_host, size_t(B * rl.record_bytes), cudaMemcpyHostToDevice, st),
        "cudaMemcpyAsync (records)");
    if (rc != NEST_OK) return rc;
    rc = nest_solve(dims, rec_d, costs_d, plans_d, ws, ws_left, stream, opt);
    if (rc != NEST_OK) return rc;
    // one copy back: every plan header carries its instance's t_batch (-1 unless solved),
    // which is what costs_out holds
    if ((rc = cuda_status(cudaMemcpyAsync(plans_host, plans_d, size_t(B * plan_bytes(g)), cudaMemcpyDeviceToHost, st),
                          "cudaMemcpyAsync (plans)")) ||
        (rc = cuda_status(cudaStreamSynchronize(st), "cudaStreamSynchronize")))
        return rc;
    const unsigned char *ph = static_cast<const unsigned char *>(plans_host);
    bool timed_out = false;
    for (int64_t b = 0; b < B; b++) {
        const nest_plan_header *h = reinterpret_cast<const nest_plan_header *>(ph + b * plan_bytes(g));
        costs_host[b] = h->t_batch;
        timed_out = timed_out || h->status == NEST_TIMED_OUT;
    }
    return timed_out ? NEST_E_TIMEOUT : NEST_OK;
}

}  // extern "C"
