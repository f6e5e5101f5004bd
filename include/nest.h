/*
 * nest.h - C ABI of the GB300 solver for the Nest placement dynamic program.
 *
 * Source of the method: "Nest: Network- and Memory-Aware Device Placement for
 * Distributed Deep Learning" (cited as Nest):
 *   §3.3 peak-memory equation   Mem(S, s) = sum(2 weights + optimizer states +
 *                               activations) + (s - 1) stashed data, 1F1B positions;
 *   §4 Eq. 3                    dp[l][D][k][s] = min over D', a of
 *                               max(dp[l'][D'][k - a][s - 1], load_l(D \ D', a, s));
 *   §4 load()                   compute + tiered collectives + forward/backward link
 *                               traffic, with ZeRO and recompute in the transition;
 *   Appendix K Algorithm 1      backward sweep, t_batch = t_stage (mbs + s - 1),
 *                               stage reconstruction.
 *
 * One problem ("instance") is a chain of L layers, or a DAG of L layers (graph
 * instances, below), a cluster of D devices grouped in tiers, C candidate tiers for
 * links between pipeline stages, S parallel strategies (TP t, context-parallel cp,
 * expert-parallel e, ZeRO stage z, recompute r) and a per-device memory budget.
 * The solver returns, per instance, the smallest iteration time and a plan of
 * stages, each with a device count unit * 2^m, a strategy and the candidate tier
 * of its outgoing link.
 *
 * Graph instances (Nest §4 states Eq. 3 over downsets of the operator graph): the
 * layers are numbered topologically and succ[l] has bit v set for each edge
 * l -> v.  The DP states are the up-sets of the graph (sets closed under
 * successors: the layers not yet placed), ordered by size descending and then by
 * mask ascending - state 0 is the whole graph, the last state the empty set; a
 * chain gets its suffixes [i, L) as states i.  A stage goes from state i to a
 * state j strictly inside it and holds the layers states[i] \ states[j].  The
 * bytes entering a state (outputs of the layers outside it that feed it; for the
 * whole graph, the source layers' outputs) are its link volume and the stashed
 * input of the stage that starts there; for a chain that is ao[i - 1] (ao[0] at
 * i = 0), as in the chain model.
 * All times are int64 nanoseconds and every result is exact: the CUDA path and
 * the plain CPU definition agree bit for bit.
 *
 * Memory ownership: the caller allocates every buffer.  The library allocates
 * nothing, frees nothing and keeps no state between calls.  nest_solve only
 * enqueues work on the caller's stream; results are valid once the stream has
 * synchronised.  nest_solve_host is synchronous.
 */
#ifndef NEST_H
#define NEST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- call status (return value) ------------------------------------------ */
#define NEST_OK           0
#define NEST_E_INVALID   -1  /* null pointer, negative count or malformed argument */
#define NEST_E_LIMITS    -2  /* a batch dimension beyond the limits below */
#define NEST_E_WORKSPACE -3  /* workspace smaller than nest_workspace_size() or misaligned */
#define NEST_E_CUDA      -4  /* a CUDA runtime call failed (launch, copy, attribute) */
#define NEST_E_TIMEOUT   -5  /* nest_solve_host only: a device wait gave up (see NEST_TIMED_OUT) */

/* ---- per-instance status (nest_plan.status) -------------------------------- */
#define NEST_SOLVED     0  /* plan and t_batch valid */
#define NEST_INFEASIBLE 1  /* no plan fits memory, or every plan's bottleneck >= 2^40-1 ns */
#define NEST_BAD_INPUT  2  /* the instance breaks a rule listed under nest_record_header */
#define NEST_TIMED_OUT  3  /* a bounded wait inside the DP sweep gave up; result unusable */

/* ---- batch dimensions ------------------------------------------------------
 * Fixed strides of the instance records and of the workspace.  Limits (checked
 * on the host before any launch, NEST_E_LIMITS otherwise):
 *   1 <= Lmax <= 255 layers, 1 <= Tmax <= 8 tiers, 1 <= Cmax <= 15 candidates,
 *   1 <= Smax <= 4095 strategies, 1 <= Pcap <= 31 stages,
 *   1 <= Dumax <= 512 device units, 0 <= Vmax <= 255.
 * The DP runs over states 0 .. N per instance, N = max(Lmax, Vmax).          */
typedef struct {
    int32_t B;      /* instances in the batch (0 is a no-op) */
    int32_t Lmax;
    int32_t Tmax;
    int32_t Cmax;
    int32_t Smax;
    int32_t Pcap;
    int32_t Dumax;  /* largest D / unit of any instance */
    int32_t Vmax;   /* at least the number of non-empty up-sets of every graph instance's
                       layer graph (its DP states less the empty set); 0 when every
                       instance is a chain */
} nest_dims;

/* ---- instance record ---------------------------------------------------------
 * B records back to back, each nest_record_bytes() long, 256-byte aligned.  A
 * record starts with this header; the arrays follow at the offsets returned by
 * nest_record_layout().  Units: flops, bytes, bytes per microsecond,
 * nanoseconds, flop per nanosecond.
 * Rules (else the instance gets NEST_BAD_INPUT):
 *   1 <= L <= Lmax; unit a power of two; unit <= D <= 8192; D % unit == 0;
 *   D / unit <= Dumax; 1 <= T <= Tmax; tier sizes G strictly increasing powers of
 *   two with G[T-1] >= D; 1000 <= bw <= 2^40; 0 <= lat <= 2^24; 1 <= C <= Cmax;
 *   candidate tiers strictly increasing in [0, T); 1 <= S <= Smax; t, cp, e powers
 *   of two <= 8192; z in 0..3; r in 0..1; 1 <= Pmax <= Pcap; Pmax <= M <= 2^20;
 *   schedule in {0, 1}; graph in {0, 1};
 *   graph instances: L <= 63, every succ[l] has bits only in (l, L), and the graph
 *   has at most Vmax non-empty up-sets;
 *   1 <= R <= 2^40; 0 <= budget <= 2^62; 0 <= opt_factor <= 16; per layer
 *   0 <= fl <= 2^48, 0 <= pd, pe, ao, aw, a2a <= 2^38, moe in {0, 1}.       */
typedef struct {
    int32_t L;          /* layers */
    int32_t D;          /* devices */
    int32_t unit;       /* device counts are unit * 2^m */
    int32_t T;          /* tiers */
    int32_t C;          /* candidate tiers for inter-stage links */
    int32_t S;          /* strategies */
    int32_t Pmax;       /* largest number of pipeline stages */
    int32_t schedule;   /* 0 = 1F1B (a stage at position p from the end stashes p - 1
                           microbatches), 1 = GPipe (each of the q data-parallel replicas
                           of a stage holds all its ceil(M / q) microbatches) */
    int64_t R;          /* device compute rate, flop per ns */
    int64_t M;          /* microbatches per iteration */
    int64_t budget;     /* bytes per device */
    int64_t opt_factor; /* optimizer-state bytes per bf16 weight byte */
    int32_t graph;      /* 0 = chain 0 -> 1 -> ... -> L-1 (succ ignored), 1 = the DAG in succ */
    int32_t reserved;
} nest_record_header;

/* Byte offsets inside one record (from its start). */
typedef struct {
    int64_t record_bytes; /* stride between records (multiple of 256) */
    int64_t fl, pd, pe, ao, aw, a2a; /* int64 [Lmax] each */
    int64_t moe;                     /* uint8 [Lmax] */
    int64_t G, bw, lat;              /* int64 [Tmax] each */
    int64_t cand;                    /* int32 [Cmax] */
    int64_t strat;                   /* int16 [Smax][8]: t, cp, e, z, r, 0, 0, 0 */
    int64_t succ;                    /* uint64 [Lmax]: successor masks (graph instances) */
} nest_layout;

/* ---- output plan --------------------------------------------------------------
 * B plan records back to back, each nest_plan_bytes() long: a nest_plan_header
 * followed by Pcap nest_stage entries (n_stages of them used).               */
typedef struct {
    int16_t i, j;    /* the stage goes from DP state i to state j: layers [i, j) of a chain,
                        states[i] \ states[j] of a graph (state order above) */
    int16_t s;       /* strategy index into the instance's strategy table */
    int8_t c_next;   /* candidate of the link to the next stage, -1 for the last stage */
    int8_t reserved;
    int32_t k;       /* devices of the stage */
    int32_t reserved2;
    uint64_t layers; /* bit l set for each layer of the stage (0 for chains of more than
                        64 layers) */
} nest_stage;

typedef struct {
    int32_t status;     /* NEST_SOLVED .. NEST_TIMED_OUT */
    int32_t n_stages;
    int64_t t_batch;    /* iteration time in ns, -1 unless solved */
    int64_t bottleneck; /* largest stage time per microbatch in ns, -1 unless solved */
} nest_plan_header;

/* ---- options -------------------------------------------------------------------
 * Zero-initialised options (or a NULL pointer) select the defaults.            */
typedef struct {
    int32_t chunk;          /* instances per pass through the kernels; 0 = all, at most 65535 (the
                               workspace must be sized for the same chunk) */
    int32_t sweep_cluster;  /* CTAs per instance in the DP sweep: 0 = auto, or 1, 2, 4, 8, 16 */
    int32_t sweep_jsplit;   /* threads sharing one DP cell: 0 = auto, or 1, 2, 4, 8, as long as
                               the CTA stays within 512 threads (else NEST_E_INVALID) */
    int32_t sweep_variant;  /* 0 = auto; 1 = rows resident in shared memory (NEST_E_LIMITS
                               if they do not fit, or with sweep_cluster 1 when Pcap > 1:
                               rows go to the next position's CTA, which must be another
                               one); 2 = rows streamed from global memory (64-bit words);
                               3 = layered: one launch per pipeline position over every
                               instance, 32-bit tagged words (NEST_E_LIMITS beyond four
                               candidates; instances whose values the words cannot hold
                               are solved again by a streaming launch of the same call).
                               The choice changes no result. */
    int64_t spin_limit;     /* polls before a device wait gives up (each poll suspends for at
                               most 20 us): 0 = default (2^16, about a second); a negative
                               value makes every wait give up at once, which exercises the
                               timeout path (instances end NEST_TIMED_OUT) */
    void **events;          /* optional cudaEvent_t[5 * chunks]; for chunk n, events
                               [5n .. 5n+4] are recorded on the stream before prep, the stage
                               loads (cost build and strategy reduction), DP sweep and
                               backtrack, and after backtrack.  NULL = no events; NULL
                               entries are skipped.  The kernels otherwise launch with
                               programmatic dependent launch (each may be scheduled while its
                               predecessor finishes); an event between two of them
                               serialises that boundary. */
    uint32_t flags;         /* NEST_KEEP_COSTS, or 0 */
    int32_t reserved;
} nest_options;

/* Also write the stage-cost tensor (every (stage, width, strategy) word, before the
 * per-position strategy minimum) into the workspace, for inspection.  The solve does
 * not need it; the workspace must then hold nest_workspace_size_costs() bytes. */
#define NEST_KEEP_COSTS 1u

/* Fills *out with the record layout for dims.  Returns NEST_OK or NEST_E_LIMITS. */
int nest_record_layout(const nest_dims *dims, nest_layout *out);

/* Stride of one plan record in bytes (0 when dims break the limits). */
size_t nest_plan_bytes(const nest_dims *dims);

/* Device workspace bytes that nest_solve needs for passes of `chunk` instances
 * (chunk <= 0 means dims->B).  0 when dims break the limits.  The workspace holds,
 * per instance of a chunk, the derived per-instance tables, the per-position
 * strategy loads, the DP value and argument tables and a 32-bit copy of the values
 * (read by the layered sweep). */
size_t nest_workspace_size(const nest_dims *dims, int32_t chunk);

/* The same plus room for the stage-cost tensor cost[pair(i, j)][m][s] (8 bytes per
 * word): what nest_solve needs with NEST_KEEP_COSTS. */
size_t nest_workspace_size_costs(const nest_dims *dims, int32_t chunk);

/* Solve a batch on the GPU.
 *   records    DEVICE, B instance records (layout above), read only
 *   costs_out  DEVICE int64 [B]: t_batch per instance, -1 unless NEST_SOLVED
 *   plans_out  DEVICE, B plan records of nest_plan_bytes() each
 *   workspace  DEVICE, >= nest_workspace_size(dims, opt->chunk) bytes, 256-byte aligned;
 *              contents on entry are ignored, on return undefined
 *   stream     a cudaStream_t (NULL = legacy default stream)
 * Instances are independent; a bad instance only sets its own status.  Returns
 * NEST_OK once every kernel is enqueued; NEST_E_* (nothing enqueued) on bad
 * arguments; NEST_E_CUDA if a launch fails. */
int nest_solve(const nest_dims *dims, const void *records, int64_t *costs_out, void *plans_out,
               void *workspace, size_t ws_bytes, void *stream, const nest_options *opt);

/* Device workspace bytes for nest_solve_host: nest_workspace_size plus room for
 * the records and the results. */
size_t nest_workspace_size_host(const nest_dims *dims, int32_t chunk);

/* Solve a batch held in HOST memory: copies the records to the device workspace,
 * solves, copies the plans back (costs_host is filled from their headers' t_batch)
 * and synchronises the stream.
 *   records_host, costs_host, plans_host   HOST buffers (pinned memory is faster)
 *   workspace    DEVICE, >= nest_workspace_size_host(dims, opt->chunk) bytes
 * Returns NEST_OK, NEST_E_TIMEOUT if some instance timed out, or NEST_E_*. */
int nest_solve_host(const nest_dims *dims, const void *records_host, int64_t *costs_host,
                    void *plans_host, void *workspace, size_t ws_bytes, void *stream,
                    const nest_options *opt);

/* Offsets (bytes from the workspace start) of the intermediate tables of the
 * LAST chunk a nest_solve call processed, for inspection after the stream syncs:
 *   loads uint64 [chunk][Pcap][NP][Kpad]  (tau* << 16) | s* per position p (index p-1)
 *   dpv   int64  [chunk][Pcap][N][Cmax][Dpad]  DP value per (p, i, c, d), 2^40-1 = none
 *   dpa   uint32 [chunk][Pcap][N][Cmax][Dpad]  (j << 8) | (m << 4) | c'
 *   cost  uint64 [chunk][NP][Kmax][Spad]  (tau << 8) | pmax, all ones = not applicable;
 *         written only with NEST_KEEP_COSTS, after the end of the plain workspace
 * where NP = N (N + 1) / 2 pairs of states (i, j) ordered by i then j (for a graph
 * instance the pairs whose state j is not inside state i hold all
 * ones), Kmax =
 * floor(log2 Dumax) + 1, Kpad = Kmax rounded up to even, Spad = Smax rounded up
 * to even, Dpad = Dumax + 1 rounded up to a multiple of 4.  total and total_costs
 * are nest_workspace_size and nest_workspace_size_costs. */
typedef struct {
    int64_t loads, dpv, dpa, cost, total, total_costs;
    int32_t NP, Kmax, Kpad, Spad, Dpad, chunk, N, reserved;
} nest_ws_layout;
int nest_workspace_layout(const nest_dims *dims, int32_t chunk, nest_ws_layout *out);

/* ---- launch description ----------------------------------------------------------
 * What nest_solve launches for these dims and options on the current device, without
 * launching anything: the passes, the kernels of a pass and the DP-sweep shape.  The
 * sweep shape follows the device's shared memory and occupancy, so call it with the
 * device current that will run the solve.  When the resident sweep sized for 32-bit
 * value words alone (instances whose largest load plus two link costs stays below
 * 2^30 ns; for a graph instance in a batch of at most two link candidates, at most
 * 2^(32 - b) - 2 ns, b = 2, 3 or 4 for up to 4, 8 or 16 widths) needs fewer waves than
 * one sized for both widths, the sweep is split: that launch takes the 32-bit instances
 * and a second launch the others.
 * Returns NEST_OK, NEST_E_INVALID (null pointer, bad option) or NEST_E_LIMITS. */
typedef struct {
    int32_t chunks;             /* passes through the kernels */
    int32_t kernels_per_chunk;  /* launches per pass: prep, stage loads, the sweep (1 or 2 resident
                                   or streaming launches; layered: 1 + 2 (Pcap - 1) + 1), backtrack */
    int32_t sweep_variant;      /* 1 = rows resident in shared memory, 2 = streamed from global
                                   memory, 3 = layered (one launch per position and tag mode) */
    int32_t sweep_cluster;      /* CTAs per instance */
    int32_t sweep_jsplit;       /* threads per DP cell */
    int32_t sweep_threads;      /* threads per CTA */
    int32_t sweep_split;        /* 1: a second sweep launch (wide_*) takes the 64-bit-word instances */
    int32_t wide_variant, wide_cluster, wide_jsplit, wide_threads;
    int32_t reserved;
} nest_launch_desc;
int nest_describe_launch(const nest_dims *dims, const nest_options *opt, nest_launch_desc *out);

/* ---- joint search over variants -------------------------------------------------
 * Nest §5.2.3 explores the microbatch size together with the placement.  The
 * variants of a problem (e.g. the same model with 1, 2, 4 and 8 samples per
 * microbatch, M scaled to keep the global batch) are solved as consecutive
 * instances of one batch; this picks, per group of `group` consecutive instances,
 * the index within the group of the smallest t_batch, ties to the smaller index, -1
 * when no variant is solved.
 *   costs     DEVICE int64 [B], as written by nest_solve (may be the same stream's
 *             output: the call is ordered after it on `stream`)
 *   best_out  DEVICE int32 [B / group]
 * Returns NEST_OK once the kernel is enqueued, NEST_E_INVALID when group < 1 or B is
 * not a multiple of group, NEST_E_CUDA if the launch fails. */
int nest_select_best(const int64_t *costs, int32_t B, int32_t group, int32_t *best_out, void *stream);

/* ---- solve without allocation ------------------------------------------------
 * No counterpart in the paper: this serves callers that cannot allocate device
 * memory - a serving or scheduling process that has handed all device memory to its
 * own pool, a plug-in inside a host application that forbids device allocations in
 * its callbacks, code that must not stall on the device-wide synchronisation that
 * cudaMalloc / cudaFree can cause.
 *
 * Same arguments and results as nest_solve, without the workspace: the scratch
 * memory is a fixed array of NEST_STATIC_SCRATCH_BYTES inside the library, held by
 * every GPU that loads the library until the process exits.  The call allocates
 * nothing and frees nothing.  Returns NEST_E_WORKSPACE when the batch (or chunk,
 * opt->chunk) needs more scratch than that - nest_workspace_size() tells how much -,
 * NEST_E_INVALID with NEST_KEEP_COSTS (the stage-cost tensor would land in the array,
 * out of the caller's reach), and otherwise what nest_solve returns.  A call made
 * outside a stream capture looks up the array's device address for the current device
 * (so a device reset does not leave a stale address behind); a call made while its
 * stream is being captured reuses the address of the last such lookup on that device,
 * so make one call before capturing (else NEST_E_INVALID).  All calls share the array
 * and it keeps the last call's contents (nothing in it needs clearing: the solve
 * writes every scratch word before reading it); calls whose work overlaps on the GPU
 * race on it, so the caller must serialise them (one stream, or an event between
 * them). */
#define NEST_STATIC_SCRATCH_BYTES (64u << 20)
int nest_solve_static(const nest_dims *dims, const void *records, int64_t *costs_out, void *plans_out,
                      void *stream, const nest_options *opt);

#ifdef __cplusplus
}
#endif
#endif /* NEST_H */
