"""Mutation check of the oracle's pins (run by hand: `python tests/oracle_mutations.py`).

The oracle is trusted because its CPU tests pin it to closed forms, brute force,
textbook special cases and invariants.  This script checks that those pins would
notice a plausible mistake: it plants one mistake at a time in a scratch copy of
`oracle/nest_oracle.c` (a floored ceiling, a collective priced on the wrong group,
tier, count or volume, a term left out of the stage time or the memory, ZeRO
sharding at the wrong stage, an off-by-one in pmax, the pipeline bubble or the stash
index, the width rule, a dropped link cost, the wrong tie-break, an inclusive cap, a
relaxed validation bound, the up-set order or link volumes of a layer graph), runs
the oracle's pin tests against that copy, and reports each mistake as caught or
survived.  The stored results of the mixed 128-layer workload are left out: they
were written by the oracle itself, so they pin nothing about it.

Exit status 0 when every mistake is caught.  About 20 minutes on 8 cores.
"""
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["test_oracle_brute.py", "test_oracle_costmodel.py", "test_oracle_gpipe.py",
        "test_oracle_invariants.py", "test_oracle_joint.py", "test_oracle_lattice.py",
        "test_oracle_special.py", "test_synth_torus.py"]

# (what the mistake is, the text it replaces, the replacement); the first occurrence
# is replaced (the chain solver's, where the layer-graph solver repeats a line).
MUTATIONS = [
    ("ceiling division floors", "return a / b + (a % b != 0);", "return a / b;"),
    ("collective latency steps lose phi", "cnt * phi * (n - 1) * x->lat[tr]", "cnt * (n - 1) * x->lat[tr]"),
    ("collective moves the whole volume", "cdiv(phi * (n - 1) * V, n)", "(phi * V)"),
    ("transfer time without the ns/us factor", "cdiv(per_device * 1000, x->bw[tr])", "cdiv(per_device, x->bw[tr])"),
    ("tier choice off by one", "while (x->G[t] < n) t++;", "while (x->G[t] <= n && t < x->T - 1) t++;"),
    ("recompute costs two passes", "u->Fl * (3 + rc), t * cp * x->R", "u->Fl * (3 + 2 * rc), t * cp * x->R"),
    ("compute not split by cp", "u->Fl * (3 + rc), t * cp * x->R", "u->Fl * (3 + rc), t * x->R"),
    ("backward pass costs one forward", "u->Fl * (3 + rc), t * cp * x->R", "u->Fl * (2 + rc), t * cp * x->R"),
    ("TP volume not split by cp", "4 * cdiv(u->Ao, cp), 4 * u->nL", "4 * u->Ao, 4 * u->nL"),
    ("TP priced on the stage's tier", "coll(x, 2, t, tier_of(x, t),", "coll(x, 2, t, tk,"),
    ("TP two AllReduces per layer", "tier_of(x, t), 4 * cdiv(u->Ao, cp), 4 * u->nL", "tier_of(x, t), 2 * cdiv(u->Ao, cp), 2 * u->nL"),
    ("TP AllReduce priced as AllGather", "r->tp = coll(x, 2, t,", "r->tp = coll(x, 1, t,"),
    ("CP volume not split by t", "4 * cdiv(u->Ao, t), 4 * u->nL", "4 * u->Ao, 4 * u->nL"),
    ("CP priced on the tier of cp", "coll(x, 1, cp, tier_of(x, t * cp),", "coll(x, 1, cp, tier_of(x, cp),"),
    ("EP volume not split by cp", "4 * cdiv(u->A2, t * cp), 4 * u->nM", "4 * cdiv(u->A2, t), 4 * u->nM"),
    ("EP steps counted per layer", "4 * cdiv(u->A2, t * cp), 4 * u->nM", "4 * cdiv(u->A2, t * cp), 4 * u->nL"),
    ("EP priced on the tier of e", "coll(x, 1, e, tier_of(x, t * cp * e),", "coll(x, 1, e, tier_of(x, e),"),
    ("ZeRO-3 gathers once", "coll(x, 1, q, tk, 2 * Wd, 2 * u->nL)", "coll(x, 1, q, tk, Wd, u->nL)"),
    ("ZeRO-3 expert gathers over q", "coll(x, 1, qe, tk, 2 * We, 2 * u->nM)", "coll(x, 1, q, tk, 2 * We, 2 * u->nM)"),
    ("ZeRO-3 expert gathers left out", "+ coll(x, 1, qe, tk, 2 * We, 2 * u->nM);", ";"),
    ("ZeRO-0 sync as ReduceScatter", "r->sd = coll(x, 2, q, tk, Wd, u->nL);", "r->sd = coll(x, 1, q, tk, Wd, u->nL);"),
    ("expert sync over q", "r->se = coll(x, 2, qe, tk, We, u->nM);", "r->se = coll(x, 2, q, tk, We, u->nM);"),
    ("ZeRO-3 sync adds an AllGather", "int64_t mult = z < 3 ? 2 : 1;", "int64_t mult = 2;"),
    ("ZeRO-2 sync without the AllGather", "int64_t mult = z < 3 ? 2 : 1;", "int64_t mult = z < 2 ? 2 : 1;"),
    ("stage time without EP", "r->comp + r->tp + r->cpc + r->ep + r->z3, q", "r->comp + r->tp + r->cpc + r->z3, q"),
    ("sync not amortised over M", "cdiv(r->sd + r->se, x->M)", "(r->sd + r->se)"),
    ("stage time without the expert sync", "cdiv(r->sd + r->se, x->M)", "cdiv(r->sd, x->M)"),
    ("replica time not divided by q", "cdiv(r->comp + r->tp + r->cpc + r->ep + r->z3, q)", "(r->comp + r->tp + r->cpc + r->ep + r->z3)"),
    ("dense weights not split by t", "int64_t Wd = cdiv(u->Pd, t);", "int64_t Wd = u->Pd;"),
    ("expert weights not split by e", "int64_t We = cdiv(u->Pe, t * e);", "int64_t We = cdiv(u->Pe, t);"),
    ("weights sharded from ZeRO-2", "r->w = z == 3 ?", "r->w = z >= 2 ?"),
    ("gradients sharded from ZeRO-1", "r->g = z >= 2 ?", "r->g = z >= 1 ?"),
    ("optimizer states sharded from ZeRO-2", "r->o = z >= 1 ?", "r->o = z >= 2 ?"),
    ("expert states sharded over q", "cdiv(Wd, q) + cdiv(We, qe) : Wd + We;\n    r->g", "cdiv(Wd, q) + cdiv(We, q) : Wd + We;\n    r->g"),
    ("activations not split by cp", "r->act = cdiv(rc ? u->AwMax : u->Aw, t * cp);", "r->act = cdiv(rc ? u->AwMax : u->Aw, t);"),
    ("activations left out of the static memory", "r->stat = r->w + r->g + r->o + r->act;", "r->stat = r->w + r->g + r->o;"),
    ("recompute keeps every activation", "r->act = cdiv(rc ? u->AwMax : u->Aw, t * cp);", "r->act = cdiv(u->Aw, t * cp);"),
    ("recompute stashes every activation", "r->stash = cdiv(rc ? u->ain : u->Aw, t * cp);", "r->stash = cdiv(u->Aw, t * cp);"),
    ("optimizer states lose their factor", ": opt * (Wd + We);", ": (Wd + We);"),
    ("GPipe holds all M microbatches", "/ cdiv(x->M, q) ? x->Pmax : 0;", "/ x->M ? x->Pmax : 0;"),
    ("pmax off by one", "imin(x->Pmax, 1 + (x->budget - r->stat) / r->stash)", "imin(x->Pmax, (x->budget - r->stat) / r->stash)"),
    ("stashed input is the stage's own output", "u->ain = i > 0 ? x->ao[i - 1] : x->ao[0];", "u->ain = x->ao[i];"),
    ("link carries the next layer's output", "cdiv(x->ao[b - 1] * 1000, x->bw[tr])", "cdiv(x->ao[b] * 1000, x->bw[tr])"),
    ("link without latency", "v = x->lat[tr] + cdiv(x->ao[b - 1] * 1000, x->bw[tr]);", "v = cdiv(x->ao[b - 1] * 1000, x->bw[tr]);"),
    ("width rule k <= G", "if (i > 0 && 2 * k > x->G[x->cand[c]]) continue;", "if (i > 0 && k > x->G[x->cand[c]]) continue;"),
    ("no width rule on the outgoing link", "if (2 * k > x->G[x->cand[c2]]) continue;", ";"),
    ("outgoing link cost left out", "imax(base + X[j * C + c2], (int64_t)(prev >> 24))", "imax(base, (int64_t)(prev >> 24))"),
    ("incoming link cost left out", "const int64_t base = tstar + (i > 0 ? X[i * C + c] : 0);", "const int64_t base = tstar;"),
    ("stage times added instead of maximised", "imax(base + X[j * C + c2], (int64_t)(prev >> 24))", "(base + X[j * C + c2] + (int64_t)(prev >> 24))"),
    ("bubble off by one", "(int64_t)(key >> 24) * (x->M + p - 1)", "(int64_t)(key >> 24) * (x->M + p)"),
    ("no bubble", "(int64_t)(key >> 24) * (x->M + p - 1)", "(int64_t)(key >> 24) * x->M"),
    ("batch-time ties to more stages", "if (bp < 0 || t < bt) {", "if (bp < 0 || t <= bt) {"),
    ("a load serves one position too few", "for (int p = 1; p <= pm; p++)", "for (int p = 1; p < pm; p++)"),
    ("strategy ties to the larger index", "uint64_t key = ((w >> 8) << 16) | (uint64_t)s;", "uint64_t key = ((w >> 8) << 16) | (uint64_t)(0xFFFF - s);"),
    ("EP allowed without a MoE layer", "if (e > 1 && u->nM == 0) return;", ";"),
    ("expert degree need not divide q", "if (q % e) return;", ";"),
    ("a load at the cap is feasible", "if (!r->valid || r->tau >= OR_CAP) return OR_INF;", "if (!r->valid || r->tau > OR_CAP) return OR_INF;"),
    ("a stage time at the cap is feasible", "if (v >= OR_CAP) continue;", "if (v > OR_CAP) continue;"),
    ("a last stage at the cap is feasible", "if (base < OR_CAP) {", "if (base <= OR_CAP) {"),
    ("graph link volume from inside the set", "} else if (!(D & bit) && (succ[l] & D)) {", "} else if ((D & bit) && (succ[l] & ~D)) {"),
    ("graph entry volume from every layer", "if (src) b += x->ao[l];", "b += x->ao[l];"),
    ("up-sets ordered by ascending size", "while (b > 0 && (popc(states[b - 1]) < popc(v) ||", "while (b > 0 && (popc(states[b - 1]) > popc(v) ||"),
    ("graph stash from the set after the stage", "mask_sums(x, D & ~Dp, bytes_in(x, succ, D, all), &u);\n    for", "mask_sums(x, D & ~Dp, bytes_in(x, succ, Dp, all), &u);\n    for"),
    ("bandwidth floor not checked", "x->bw[t] < 1000 ||", "x->bw[t] < 1 ||"),
    ("M >= Pmax not checked", "if (x->M < x->Pmax ||", "if (x->M < 1 ||"),
]


def main() -> int:
    src = open(os.path.join(ROOT, "oracle", "nest_oracle.c")).read()
    work = tempfile.mkdtemp(prefix="oracle_mutations_")
    try:
        ign = shutil.ignore_patterns("__pycache__", "*.so", "_build", "*.tmp")
        for d in ("oracle", "tests", "memory_aware_device_gb300"):
            shutil.copytree(os.path.join(ROOT, d), os.path.join(work, d), ignore=ign)
        target = os.path.join(work, "oracle", "nest_oracle.c")
        survived = []
        for name, old, new in MUTATIONS:
            if old not in src:
                print(f"{name}: text not found", flush=True)
                survived.append(name)
                continue
            open(target, "w").write(src.replace(old, new, 1))
            lib = os.path.join(work, "oracle", "libnest_oracle.so")
            if os.path.exists(lib):
                os.remove(lib)   # rebuilt from the planted source by the first test
            r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] +
                               [os.path.join("tests", f) for f in PINS],
                               cwd=work, capture_output=True, text=True)
            first = next((line[7:].split(" - ")[0] for line in r.stdout.splitlines() if line.startswith("FAILED")),
                         f"a crash of the test process (exit status {r.returncode})")
            print(f"{name}: {'caught by ' + first if r.returncode else 'SURVIVED'}", flush=True)
            if r.returncode == 0:
                survived.append(name)
        print(f"{len(MUTATIONS) - len(survived)} of {len(MUTATIONS)} mistakes caught")
        return 1 if survived else 0
    finally:
        shutil.rmtree(work, ignore_errors=True)


if __name__ == "__main__":
    sys.exit(main())
