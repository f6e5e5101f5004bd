/*
 * CPU oracle for the Nest placement dynamic program.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header or table with the CUDA library.
 *
 * Source: "Nest: Network- and Memory-Aware Device Placement for Distributed Deep
 * Learning" (cited below as Nest):
 *   - §3.3, peak-memory equation: Mem(S, s) = sum over the stage's layers of
 *     (2 weights + optimizer states + activations) + (s - 1) stashed data, where s
 *     is the stage's position counted from the end of a 1F1B pipeline;
 *   - §3.3, recompute: only the stage input is stashed, at the price of one more
 *     forward pass;
 *   - §3.3, schedule: the stashed count is (s - 1) under 1F1B and scales with B/d
 *     under GPipe;
 *   - §4, Eq. 3: dp[l][D][k][s] = min over cut D' and device count a of
 *     max(dp[l'][D'][k - a][s - 1], load_l(D \ D', a, s)), solved backward over
 *     the layer suffix D, with the tier l of the (not yet placed) producer stage
 *     as a state variable ("delayed forward cost");
 *   - §4, load(): compute latency scaled by the tensor/expert degree, collective
 *     costs per network tier, forward traffic from tier l and backward traffic to
 *     D', ZeRO and recompute folded into the transition;
 *   - Appendix K, Algorithm 1: the sweep over suffixes, the final batch-time loop
 *     t_batch = t_stage * (mbs + s - 1) and the stage reconstruction.
 *
 * Readings where the pages leave a step open (each also listed in the design notes):
 *   - the layer graph is a chain, D a suffix [i, L), the cut D' the suffix [j, L);
 *   - device counts are unit * 2^m; dp[i][d][p][c] uses AT MOST d units;
 *   - c is the candidate tier of the link into the stage that starts at i; the
 *     stage that ends at j minimises over the candidate c' of the link out of it;
 *   - a link over candidate c costs lat + ceil(bytes * 1000 / bw) on each side and
 *     needs 2k <= G[cand c] for both adjacent stage widths k;
 *   - strategies (t, cp, e, z, r) are chosen per stage; q = k / (t cp) is the
 *     data-parallel degree, experts are data-parallel over q / e;
 *   - collectives follow the ring cost model: phi (n-1) latency steps per call and
 *     phi (n-1)/n of the volume per device, phi = 2 for AllReduce, else 1; a group
 *     of one device or a zero-byte volume issues no collective;
 *   - stage time per microbatch = ceil(replica time / q) + ceil(gradient sync / M);
 *   - GPipe (B/d): each of the q data-parallel replicas runs ceil(M / q) of the M
 *     microbatches and holds all of them at once, at every position; the bubble, and
 *     so the time model, is the same as for 1F1B;
 *   - SYNCCOST is folded into each stage's amortised gradient sync term;
 *   - ties: smallest (v, j, m, c') per cell, smallest (tau, s) per strategy choice,
 *     smallest (t_batch, p) at the end;
 *   - a layer DAG numbered topologically: D an up-set (closed under successors), the
 *     cut D' an up-set strictly inside D; states ordered by size descending, then
 *     by mask, so a chain gets the suffix indices; the bytes entering D are the
 *     outputs of the layers outside D that feed it (for the whole graph, the
 *     source layers' outputs) and are both the link volume and the stashed input.
 * Every function below is pinned by the CPU tests (closed forms, brute force,
 * textbook special cases and invariants).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_CAP ((int64_t)((1LL << 40) - 1))
#define OR_INF UINT64_MAX

typedef struct {
    int32_t L, D, unit, T, C, S, Pmax, schedule; /* schedule: 0 = 1F1B, 1 = GPipe */
    int64_t R, M, budget, opt_factor;
    const int64_t *fl, *pd, *pe, *ao, *aw, *a2a;
    const uint8_t *moe;
    const int64_t *G, *bw, *lat;
    const int32_t *cand;
    const int16_t *strat; /* [S][5]: t, cp, e, z, r */
} or_instance;

typedef struct {
    int32_t i, j, k, s, c_next;
} or_stage;

/* All terms of one stage, exposed so that tests can pin each one. */
typedef struct {
    int64_t valid, comp, tp, cpc, ep, z3, sd, se, tau;
    int64_t w, g, o, act, stash, stat, pmax;
} or_terms;

typedef struct {
    int64_t Fl, Pd, Pe, Ao, Aw, A2, nL, nM, AwMax, ain;
} or_sums;

static int64_t cdiv(int64_t a, int64_t b) { return a / b + (a % b != 0); }
static int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }
static int is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

/* Smallest tier whose groups hold n devices. */
static int tier_of(const or_instance *x, int64_t n) {
    int t = 0;
    while (x->G[t] < n) t++;
    return t;
}

/* Ring-model cost of cnt collectives moving V bytes in total over a group of n
 * devices on tier tr.  A group of one, or nothing to move, issues no collective. */
static int64_t coll(const or_instance *x, int64_t phi, int64_t n, int tr, int64_t V, int64_t cnt) {
    if (n == 1 || V == 0) return 0;
    int64_t steps = cnt * phi * (n - 1) * x->lat[tr];
    int64_t per_device = cdiv(phi * (n - 1) * V, n);
    return steps + cdiv(per_device * 1000, x->bw[tr]);
}

int or_validate(const or_instance *x) {
    if (x->L < 1 || x->L > 255) return 2;
    if (!is_pow2(x->unit) || x->D < x->unit || x->D > 8192 || x->D % x->unit) return 2;
    if (x->T < 1 || x->T > 8) return 2;
    for (int t = 0; t < x->T; t++) {
        if (!is_pow2(x->G[t]) || (t > 0 && x->G[t] <= x->G[t - 1])) return 2;
        if (x->bw[t] < 1000 || x->bw[t] > (1LL << 40)) return 2;
        if (x->lat[t] < 0 || x->lat[t] > (1LL << 24)) return 2;
    }
    if (x->G[x->T - 1] < x->D) return 2;
    if (x->C < 1 || x->C > 15) return 2;
    for (int c = 0; c < x->C; c++) {
        if (x->cand[c] < 0 || x->cand[c] >= x->T) return 2;
        if (c > 0 && x->cand[c] <= x->cand[c - 1]) return 2;
    }
    if (x->S < 1 || x->S > 4095) return 2;
    for (int s = 0; s < x->S; s++) {
        const int16_t *st = x->strat + 5 * s;
        for (int f = 0; f < 3; f++)
            if (!is_pow2(st[f]) || st[f] > 8192) return 2;
        if (st[3] < 0 || st[3] > 3 || st[4] < 0 || st[4] > 1) return 2;
    }
    if (x->Pmax < 1 || x->Pmax > 31) return 2;
    if (x->schedule < 0 || x->schedule > 1) return 2;
    if (x->M < x->Pmax || x->M > (1LL << 20)) return 2;
    if (x->R < 1 || x->R > (1LL << 40)) return 2;
    if (x->budget < 0 || x->budget > (1LL << 62)) return 2;
    if (x->opt_factor < 0 || x->opt_factor > 16) return 2;
    for (int l = 0; l < x->L; l++) {
        if (x->fl[l] < 0 || x->fl[l] > (1LL << 48)) return 2;
        const int64_t *b[5] = {x->pd, x->pe, x->ao, x->aw, x->a2a};
        for (int f = 0; f < 5; f++)
            if (b[f][l] < 0 || b[f][l] > (1LL << 38)) return 2;
        if (x->moe[l] > 1) return 2;
    }
    return 0;
}

/* Per-layer metadata summed over the stage [i, j) (§3.2 graph extraction output). */
static void stage_sums(const or_instance *x, int i, int j, or_sums *u) {
    memset(u, 0, sizeof *u);
    for (int l = i; l < j; l++) {
        u->Fl += x->fl[l];
        u->Pd += x->pd[l];
        u->Pe += x->pe[l];
        u->Ao += x->ao[l];
        u->Aw += x->aw[l];
        u->A2 += x->a2a[l];
        u->nM += x->moe[l];
        u->AwMax = imax(u->AwMax, x->aw[l]);
    }
    u->nL = j - i;
    u->ain = i > 0 ? x->ao[i - 1] : x->ao[0];
}

/* load() of Eq. 3 for one strategy, and the §3.3 memory model at every position. */
static void stage_terms(const or_instance *x, const or_sums *u, int m, int s, or_terms *r) {
    memset(r, 0, sizeof *r);
    const int16_t *st = x->strat + 5 * s;
    int64_t t = st[0], cp = st[1], e = st[2], z = st[3], rc = st[4];
    int64_t k = (int64_t)x->unit << m;
    if (k % (t * cp)) return;
    int64_t q = k / (t * cp);
    if (q % e) return;
    if (e > 1 && u->nM == 0) return;
    r->valid = 1;
    int64_t qe = q / e;
    int64_t Wd = cdiv(u->Pd, t);     /* dense weight bytes per device under TP */
    int64_t We = cdiv(u->Pe, t * e); /* expert weight bytes per device under TP x EP */
    int tk = tier_of(x, k);

    /* compute: forward + two backward passes (+ one recomputed forward) */
    r->comp = cdiv(u->Fl * (3 + rc), t * cp * x->R);
    /* TP: two AllReduces forward and two backward per layer */
    r->tp = coll(x, 2, t, tier_of(x, t), 4 * cdiv(u->Ao, cp), 4 * u->nL);
    /* CP: two AllGathers forward, two ReduceScatters backward per layer */
    r->cpc = coll(x, 1, cp, tier_of(x, t * cp), 4 * cdiv(u->Ao, t), 4 * u->nL);
    /* EP: dispatch + combine AllToAll, forward and backward, per MoE layer */
    r->ep = coll(x, 1, e, tier_of(x, t * cp * e), 4 * cdiv(u->A2, t * cp), 4 * u->nM);
    /* ZeRO-3 gathers the sharded weights for the forward and the backward pass */
    if (z == 3)
        r->z3 = coll(x, 1, q, tk, 2 * Wd, 2 * u->nL) + coll(x, 1, qe, tk, 2 * We, 2 * u->nM);
    /* gradient synchronisation once per iteration: AllReduce without ZeRO,
     * ReduceScatter + AllGather for ZeRO-1/2, ReduceScatter alone for ZeRO-3 */
    if (z == 0) {
        r->sd = coll(x, 2, q, tk, Wd, u->nL);
        r->se = coll(x, 2, qe, tk, We, u->nM);
    } else {
        int64_t mult = z < 3 ? 2 : 1;
        r->sd = mult * coll(x, 1, q, tk, Wd, u->nL);
        r->se = mult * coll(x, 1, qe, tk, We, u->nM);
    }
    r->tau = cdiv(r->comp + r->tp + r->cpc + r->ep + r->z3, q) + cdiv(r->sd + r->se, x->M);

    /* §3.3: weights + gradients ("2 weights"), optimizer states, activations,
     * each sharded by the ZeRO stage; plus the stashed microbatches: (position - 1)
     * under 1F1B, all ceil(M / q) of the replica's microbatches under GPipe */
    int64_t opt = x->opt_factor;
    r->w = z == 3 ? cdiv(Wd, q) + cdiv(We, qe) : Wd + We;
    r->g = z >= 2 ? cdiv(Wd, q) + cdiv(We, qe) : Wd + We;
    r->o = z >= 1 ? cdiv(opt * Wd, q) + cdiv(opt * We, qe) : opt * (Wd + We);
    r->act = cdiv(rc ? u->AwMax : u->Aw, t * cp);
    r->stash = cdiv(rc ? u->ain : u->Aw, t * cp);
    r->stat = r->w + r->g + r->o + r->act;
    if (r->stat > x->budget)
        r->pmax = 0;
    else if (x->schedule == 1)
        r->pmax = r->stash <= (x->budget - r->stat) / cdiv(x->M, q) ? x->Pmax : 0;
    else if (r->stash == 0)
        r->pmax = x->Pmax;
    else
        r->pmax = imin(x->Pmax, 1 + (x->budget - r->stat) / r->stash);
}

void or_stage_terms(const or_instance *x, int i, int j, int m, int s, or_terms *r) {
    or_sums u;
    stage_sums(x, i, j, &u);
    stage_terms(x, &u, m, s, r);
}

/* Packed stage-cost word: (tau << 8) | pmax, or all ones when the strategy does
 * not apply to this width or tau reaches the cap. */
static uint64_t word_of(const or_terms *r) {
    if (!r->valid || r->tau >= OR_CAP) return OR_INF;
    return ((uint64_t)r->tau << 8) | (uint64_t)r->pmax;
}

static int widths(const or_instance *x) {
    int K = 0;
    while (((int64_t)1 << K) <= x->D / x->unit) K++;
    return K;
}

/* cost[pair(i, j)][m][s] with pairs ordered by i, then j = i+1 .. L. */
void or_cost_tensor(const or_instance *x, uint64_t *out) {
    int K = widths(x), S = x->S;
    int64_t pair = 0;
    for (int i = 0; i < x->L; i++)
        for (int j = i + 1; j <= x->L; j++, pair++) {
            or_sums u;
            stage_sums(x, i, j, &u);
            for (int m = 0; m < K; m++)
                for (int s = 0; s < S; s++) {
                    or_terms r;
                    stage_terms(x, &u, m, s, &r);
                    out[(pair * K + m) * S + s] = word_of(&r);
                }
        }
}

/* Link cost at boundary b (between layers b-1 and b) over candidate c; zero at
 * the ends of the chain.  Out: [L+1][C]. */
void or_links(const or_instance *x, int64_t *X) {
    for (int b = 0; b <= x->L; b++)
        for (int c = 0; c < x->C; c++) {
            int64_t v = 0;
            if (b > 0 && b < x->L) {
                int tr = x->cand[c];
                v = x->lat[tr] + cdiv(x->ao[b - 1] * 1000, x->bw[tr]);
            }
            X[b * x->C + c] = v;
        }
}

/* GETLOADOFSTAGE for one stage [i, j) and every width m and position p:
 * the smallest (tau, s) over strategies whose memory fits position p.
 * out[m * Pmax + (p - 1)] = (tau << 16) | s, or all ones. */
static void stage_loads(const or_instance *x, int i, int j, int K, uint64_t *out) {
    or_sums u;
    stage_sums(x, i, j, &u);
    for (int m = 0; m < K; m++) {
        for (int p = 1; p <= x->Pmax; p++) out[m * x->Pmax + p - 1] = OR_INF;
        for (int s = 0; s < x->S; s++) {
            or_terms r;
            stage_terms(x, &u, m, s, &r);
            uint64_t w = word_of(&r);
            if (w == OR_INF) continue;
            uint64_t key = ((w >> 8) << 16) | (uint64_t)s;
            int pm = (int)(w & 0xFF);
            for (int p = 1; p <= pm; p++)
                if (key < out[m * x->Pmax + p - 1]) out[m * x->Pmax + p - 1] = key;
        }
    }
}

/* Loads for every pair: out[(pair * K + m) * Pmax + p - 1]. */
void or_loads(const or_instance *x, uint64_t *out) {
    int K = widths(x);
    int64_t pair = 0;
    for (int i = 0; i < x->L; i++)
        for (int j = i + 1; j <= x->L; j++, pair++)
            stage_loads(x, i, j, K, out + pair * K * x->Pmax);
}

int64_t or_dp_table_words(const or_instance *x) {
    int64_t Du = x->D / x->unit;
    return (int64_t)(x->L + 1) * (Du + 1) * (x->Pmax + 1) * x->C;
}

static uint64_t pack_key(int64_t v, int j, int m, int c) {
    return ((uint64_t)v << 24) | ((uint64_t)j << 8) | ((uint64_t)m << 4) | (uint64_t)c;
}

/* Eq. 3 swept backward over suffixes (Algorithm 1), then the batch-time loop and
 * the stage reconstruction.  dp_out (optional) receives the key table
 * [(L+1)][Du+1][Pmax+1][C].  Returns 0 solved, 1 infeasible, 2 invalid input. */
int or_solve(const or_instance *x, uint64_t *dp_out, int64_t *t_batch, int64_t *bottleneck,
             int32_t *n_stages, or_stage *stages) {
    *t_batch = -1;
    *bottleneck = -1;
    *n_stages = 0;
    if (or_validate(x)) return 2;
    const int L = x->L, C = x->C, P = x->Pmax, K = widths(x);
    const int64_t Du = x->D / x->unit;
    const int64_t nd = Du + 1, np = P + 1;
#define KEY(i, d, p, c) keys[(((int64_t)(i) * nd + (d)) * np + (p)) * C + (c)]
    uint64_t *keys = dp_out ? dp_out : malloc(sizeof(uint64_t) * or_dp_table_words(x));
    int64_t *X = malloc(sizeof(int64_t) * (L + 1) * C);
    uint64_t *ld = malloc(sizeof(uint64_t) * K * P);
    for (int64_t w = 0; w < or_dp_table_words(x); w++) keys[w] = OR_INF;
    /* base case: no layers left, no stages, zero latency */
    for (int64_t d = 0; d <= Du; d++)
        for (int c = 0; c < C; c++) KEY(L, d, 0, c) = 0;
    or_links(x, X);

    for (int i = L - 1; i >= 0; i--) {
        const int ncell = i == 0 ? 1 : C; /* the first stage has no producer link */
        for (int j = i + 1; j <= L; j++) {
            stage_loads(x, i, j, K, ld);
            for (int p = 1; p <= P && p <= L - i; p++) {
                if ((j == L) != (p == 1)) continue;
                for (int64_t d = 1; d <= Du; d++)
                    for (int m = 0; ((int64_t)1 << m) <= d; m++) {
                        const int64_t k = (int64_t)x->unit << m;
                        const uint64_t load = ld[m * P + p - 1];
                        if (load == OR_INF) continue;
                        const int64_t tstar = (int64_t)(load >> 16);
                        for (int c = 0; c < ncell; c++) {
                            if (i > 0 && 2 * k > x->G[x->cand[c]]) continue;
                            const int64_t base = tstar + (i > 0 ? X[i * C + c] : 0);
                            uint64_t best = KEY(i, d, p, c);
                            if (j == L) {
                                /* last stage: the previous state is the base case (0) */
                                if (base < OR_CAP) {
                                    const uint64_t cand_key = pack_key(base, j, m, 0);
                                    if (cand_key < best) best = cand_key;
                                }
                            } else {
                                for (int c2 = 0; c2 < C; c2++) {
                                    if (2 * k > x->G[x->cand[c2]]) continue;
                                    const uint64_t prev = KEY(j, d - ((int64_t)1 << m), p - 1, c2);
                                    if (prev == OR_INF) continue;
                                    const int64_t v = imax(base + X[j * C + c2], (int64_t)(prev >> 24));
                                    if (v >= OR_CAP) continue;
                                    const uint64_t cand_key = pack_key(v, j, m, c2);
                                    if (cand_key < best) best = cand_key;
                                }
                            }
                            KEY(i, d, p, c) = best;
                        }
                    }
            }
        }
    }

    /* t_batch = t_stage * (M + p - 1), smallest (t_batch, p) */
    int bp = -1;
    int64_t bt = 0;
    for (int p = 1; p <= P && p <= L; p++) {
        const uint64_t key = KEY(0, Du, p, 0);
        if (key == OR_INF) continue;
        const int64_t t = (int64_t)(key >> 24) * (x->M + p - 1);
        if (bp < 0 || t < bt) {
            bt = t;
            bp = p;
        }
    }
    int status = 1;
    if (bp > 0) {
        status = 0;
        *t_batch = bt;
        *bottleneck = (int64_t)(KEY(0, Du, bp, 0) >> 24);
        int i = 0, p = bp, c = 0, n = 0;
        int64_t d = Du;
        while (i < L) {
            const uint64_t key = KEY(i, d, p, c);
            const int j = (int)((key >> 8) & 0xFF), m = (int)((key >> 4) & 0xF), c2 = (int)(key & 0xF);
            stage_loads(x, i, j, K, ld);
            stages[n].i = i;
            stages[n].j = j;
            stages[n].k = x->unit << m;
            stages[n].s = (int32_t)(ld[m * P + p - 1] & 0xFFFF);
            stages[n].c_next = j < L ? c2 : -1;
            n++;
            d -= (int64_t)1 << m;
            p -= 1;
            c = c2;
            i = j;
        }
        *n_stages = n;
    }
    free(ld);
    free(X);
    if (!dp_out) free(keys);
#undef KEY
    return status;
}

/* ---------------------------------------------------------------------------------
 * Non-chain layer graphs.  Nest §4 states Eq. 3 over downsets of the operator
 * graph: the DP state is the set of layers not yet placed, a stage is the
 * difference of two such sets.  Reading for a DAG whose layers are numbered
 * topologically (every edge u -> v has u < v): the states are the up-sets (closed
 * under successors), ordered by size descending and then by mask; a transition
 * goes from D to any up-set D' strictly inside D and places the stage D \ D'.  For
 * a chain the up-sets are the suffixes [i, L) with the same indices, so everything
 * below reduces to the chain solver above.
 * ------------------------------------------------------------------------------- */

#define OR_MAX_STATES 256

static int popc(uint64_t v) { return __builtin_popcountll(v); }

/* Up-sets of the DAG given by succ[l] (bit v set for each edge l -> v, v > l):
 * grown from the empty set by adding a layer whose successors are all present.
 * Returns the count, or -1 when the graph is not topologically numbered, has more
 * than 63 layers, or more than OR_MAX_STATES up-sets. */
int or_lattice_states(const or_instance *x, const uint64_t *succ, uint64_t *states) {
    const int L = x->L;
    if (L < 1 || L > 63) return -1;
    for (int l = 0; l < L; l++)
        if (succ[l] & (((uint64_t)2 << l) - 1)) return -1;   /* edges go forward */
    int n = 1;
    states[0] = 0;
    for (int q = 0; q < n; q++) {
        const uint64_t D = states[q];
        for (int l = 0; l < L; l++) {
            const uint64_t bit = (uint64_t)1 << l;
            if ((D & bit) || (succ[l] & ~D)) continue;
            const uint64_t E = D | bit;
            int seen = 0;
            for (int r = 0; r < n && !seen; r++) seen = states[r] == E;
            if (seen) continue;
            if (n == OR_MAX_STATES) return -1;
            states[n++] = E;
        }
    }
    /* size descending, then mask ascending */
    for (int a = 1; a < n; a++) {
        const uint64_t v = states[a];
        int b = a;
        while (b > 0 && (popc(states[b - 1]) < popc(v) || (popc(states[b - 1]) == popc(v) && states[b - 1] > v))) {
            states[b] = states[b - 1];
            b--;
        }
        states[b] = v;
    }
    return n;
}

/* Bytes entering up-set D: the outputs of the layers outside D that feed it; for
 * the whole graph, the outputs of its source layers. */
static int64_t bytes_in(const or_instance *x, const uint64_t *succ, uint64_t D, uint64_t all) {
    int64_t b = 0;
    for (int l = 0; l < x->L; l++) {
        const uint64_t bit = (uint64_t)1 << l;
        if (D == all) {
            int src = 1;
            for (int u = 0; u < l; u++)
                if (succ[u] & bit) src = 0;
            if (src) b += x->ao[l];
        } else if (!(D & bit) && (succ[l] & D)) {
            b += x->ao[l];
        }
    }
    return b;
}

static void mask_sums(const or_instance *x, uint64_t S, int64_t ain, or_sums *u) {
    memset(u, 0, sizeof *u);
    for (int l = 0; l < x->L; l++) {
        if (!(S >> l & 1)) continue;
        u->Fl += x->fl[l];
        u->Pd += x->pd[l];
        u->Pe += x->pe[l];
        u->Ao += x->ao[l];
        u->Aw += x->aw[l];
        u->A2 += x->a2a[l];
        u->nM += x->moe[l];
        u->AwMax = imax(u->AwMax, x->aw[l]);
        u->nL++;
    }
    u->ain = ain;
}

/* Link cost into each state over each candidate: out[state][c], zero for the whole
 * graph and for the empty set. */
static void lattice_links(const or_instance *x, const uint64_t *succ, const uint64_t *st, int ns, int64_t *X) {
    const uint64_t all = st[0];
    for (int q = 0; q < ns; q++)
        for (int c = 0; c < x->C; c++) {
            int64_t v = 0;
            if (q > 0 && q < ns - 1) {
                const int tr = x->cand[c];
                v = x->lat[tr] + cdiv(bytes_in(x, succ, st[q], all) * 1000, x->bw[tr]);
            }
            X[q * x->C + c] = v;
        }
}

static void lattice_stage_loads(const or_instance *x, const uint64_t *succ, uint64_t D, uint64_t Dp, uint64_t all,
                                int K, uint64_t *out) {
    or_sums u;
    mask_sums(x, D & ~Dp, bytes_in(x, succ, D, all), &u);
    for (int m = 0; m < K; m++) {
        for (int p = 1; p <= x->Pmax; p++) out[m * x->Pmax + p - 1] = OR_INF;
        for (int s = 0; s < x->S; s++) {
            or_terms r;
            stage_terms(x, &u, m, s, &r);
            uint64_t w = word_of(&r);
            if (w == OR_INF) continue;
            uint64_t key = ((w >> 8) << 16) | (uint64_t)s;
            int pm = (int)(w & 0xFF);
            for (int p = 1; p <= pm; p++)
                if (key < out[m * x->Pmax + p - 1]) out[m * x->Pmax + p - 1] = key;
        }
    }
}

/* Loads of every transition (i, j), i < j, states[j] strictly inside states[i],
 * in that order: out[(t * K + m) * Pmax + p - 1].  Returns the transition count. */
int64_t or_lattice_loads(const or_instance *x, const uint64_t *succ, const uint64_t *st, int ns, uint64_t *out) {
    const int K = widths(x);
    int64_t t = 0;
    for (int i = 0; i < ns; i++)
        for (int j = i + 1; j < ns; j++) {
            if ((st[j] & ~st[i]) || st[j] == st[i]) continue;
            if (out) lattice_stage_loads(x, succ, st[i], st[j], st[0], K, out + t * K * x->Pmax);
            t++;
        }
    return t;
}

/* Eq. 3 over the up-sets of the DAG (the chain solver with j ranging over the
 * states inside state i), the batch-time loop and the stage reconstruction; stage
 * i and j fields are state indices.  dp_out (optional): [ns][Du+1][Pmax+1][C].
 * Returns 0 solved, 1 infeasible, 2 invalid input (also a graph beyond the
 * lattice limits). */
int or_solve_lattice(const or_instance *x, const uint64_t *succ, uint64_t *dp_out, int64_t *t_batch,
                     int64_t *bottleneck, int32_t *n_stages, or_stage *stages) {
    *t_batch = -1;
    *bottleneck = -1;
    *n_stages = 0;
    if (or_validate(x)) return 2;
    uint64_t st[OR_MAX_STATES];
    const int ns = or_lattice_states(x, succ, st);
    if (ns < 2) return 2;
    const int C = x->C, P = x->Pmax, K = widths(x);
    const int64_t Du = x->D / x->unit;
    const int64_t nd = Du + 1, np = P + 1;
    const int E = ns - 1; /* the empty set */
#define KEY(i, d, p, c) keys[(((int64_t)(i) * nd + (d)) * np + (p)) * C + (c)]
    const int64_t words = (int64_t)ns * nd * np * C;
    uint64_t *keys = dp_out ? dp_out : malloc(sizeof(uint64_t) * words);
    int64_t *X = malloc(sizeof(int64_t) * ns * C);
    uint64_t *ld = malloc(sizeof(uint64_t) * K * P);
    for (int64_t w = 0; w < words; w++) keys[w] = OR_INF;
    for (int64_t d = 0; d <= Du; d++)
        for (int c = 0; c < C; c++) KEY(E, d, 0, c) = 0;
    lattice_links(x, succ, st, ns, X);

    for (int i = E - 1; i >= 0; i--) {
        const int ncell = i == 0 ? 1 : C;
        const int layers = popc(st[i]);
        for (int j = i + 1; j <= E; j++) {
            if ((st[j] & ~st[i]) || st[j] == st[i]) continue;
            lattice_stage_loads(x, succ, st[i], st[j], st[0], K, ld);
            for (int p = 1; p <= P && p <= layers; p++) {
                if ((j == E) != (p == 1)) continue;
                for (int64_t d = 1; d <= Du; d++)
                    for (int m = 0; ((int64_t)1 << m) <= d; m++) {
                        const int64_t k = (int64_t)x->unit << m;
                        const uint64_t load = ld[m * P + p - 1];
                        if (load == OR_INF) continue;
                        const int64_t tstar = (int64_t)(load >> 16);
                        for (int c = 0; c < ncell; c++) {
                            if (i > 0 && 2 * k > x->G[x->cand[c]]) continue;
                            const int64_t base = tstar + (i > 0 ? X[i * C + c] : 0);
                            uint64_t best = KEY(i, d, p, c);
                            if (j == E) {
                                if (base < OR_CAP) {
                                    const uint64_t cand_key = pack_key(base, j, m, 0);
                                    if (cand_key < best) best = cand_key;
                                }
                            } else {
                                for (int c2 = 0; c2 < C; c2++) {
                                    if (2 * k > x->G[x->cand[c2]]) continue;
                                    const uint64_t prev = KEY(j, d - ((int64_t)1 << m), p - 1, c2);
                                    if (prev == OR_INF) continue;
                                    const int64_t v = imax(base + X[j * C + c2], (int64_t)(prev >> 24));
                                    if (v >= OR_CAP) continue;
                                    const uint64_t cand_key = pack_key(v, j, m, c2);
                                    if (cand_key < best) best = cand_key;
                                }
                            }
                            KEY(i, d, p, c) = best;
                        }
                    }
            }
        }
    }

    int bp = -1;
    int64_t bt = 0;
    for (int p = 1; p <= P && p <= popc(st[0]); p++) {
        const uint64_t key = KEY(0, Du, p, 0);
        if (key == OR_INF) continue;
        const int64_t t = (int64_t)(key >> 24) * (x->M + p - 1);
        if (bp < 0 || t < bt) {
            bt = t;
            bp = p;
        }
    }
    int status = 1;
    if (bp > 0) {
        status = 0;
        *t_batch = bt;
        *bottleneck = (int64_t)(KEY(0, Du, bp, 0) >> 24);
        int i = 0, p = bp, c = 0, n = 0;
        int64_t d = Du;
        while (i < E) {
            const uint64_t key = KEY(i, d, p, c);
            const int j = (int)((key >> 8) & 0xFF), m = (int)((key >> 4) & 0xF), c2 = (int)(key & 0xF);
            lattice_stage_loads(x, succ, st[i], st[j], st[0], K, ld);
            stages[n].i = i;
            stages[n].j = j;
            stages[n].k = x->unit << m;
            stages[n].s = (int32_t)(ld[m * P + p - 1] & 0xFFFF);
            stages[n].c_next = j < E ? c2 : -1;
            n++;
            d -= (int64_t)1 << m;
            p -= 1;
            c = c2;
            i = j;
        }
        *n_stages = n;
    }
    free(ld);
    free(X);
    if (!dp_out) free(keys);
#undef KEY
    return status;
}

/* The terms of the stage D \ D' of a layer DAG (exposed for the pins). */
void or_lattice_terms(const or_instance *x, const uint64_t *succ, uint64_t D, uint64_t Dp, int m, int s,
                      or_terms *r) {
    uint64_t all = 0;
    for (int l = 0; l < x->L; l++) all |= (uint64_t)1 << l;
    or_sums u;
    mask_sums(x, D & ~Dp, bytes_in(x, succ, D, all), &u);
    stage_terms(x, &u, m, s, r);
}

/* Link cost into up-set D over candidate c (zero for the whole graph and the empty
 * set), exposed for the pins. */
int64_t or_lattice_link(const or_instance *x, const uint64_t *succ, uint64_t D, int c) {
    uint64_t all = 0;
    for (int l = 0; l < x->L; l++) all |= (uint64_t)1 << l;
    if (D == all || D == 0) return 0;
    const int tr = x->cand[c];
    return x->lat[tr] + cdiv(bytes_in(x, succ, D, all) * 1000, x->bw[tr]);
}

/* Stage-cost words of every pair of states (i, j), i < j, in pair order (i, then j),
 * all ones where state j is not inside state i: out[pair][m][s]. */
void or_lattice_cost_tensor(const or_instance *x, const uint64_t *succ, const uint64_t *st, int ns, uint64_t *out) {
    const int K = widths(x);
    int64_t pair = 0;
    for (int i = 0; i < ns; i++)
        for (int j = i + 1; j < ns; j++, pair++)
            for (int m = 0; m < K; m++)
                for (int s = 0; s < x->S; s++) {
                    uint64_t w = OR_INF;
                    if (!(st[j] & ~st[i])) {
                        or_terms r;
                        or_lattice_terms(x, succ, st[i], st[j], m, s, &r);
                        w = word_of(&r);
                    }
                    out[(pair * K + m) * x->S + s] = w;
                }
}
