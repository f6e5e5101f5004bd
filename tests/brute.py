"""Exhaustive enumeration of every placement plan, priced from its definition.

A plan is a sequence of contiguous stages [b_0, b_1), ..., [b_{P-1}, L) with a
width unit * 2^m, a strategy per stage and a candidate tier per internal link.
Nest (Network- and Memory-Aware Device Placement), §4 Eq. 3 and Appendix K
Algorithm 1 define the optimum as the plan minimising the bottleneck stage time
times (M + P - 1), subject to the §3.3 memory model at each stage's pipeline
position.  This module enumerates all plans of a tiny instance and returns that
minimum; it reads the stage-cost words and link costs as given tables and shares
no code with the dynamic program it checks.
"""
from __future__ import annotations

import itertools

CAP = (1 << 40) - 1
INF = (1 << 64) - 1


def stage_min_tau(words_row, pos):
    """Smallest stage time over strategies whose memory fits position pos."""
    best = None
    for w in words_row:
        w = int(w)
        if w == INF:
            continue
        tau, pmax = w >> 8, w & 0xFF
        if pmax >= pos and (best is None or tau < best):
            best = tau
    return best


def enumerate_plans(inst, words, X):
    """Yield (t_batch, P, bottleneck, stages) for every feasible plan.

    words: [pair][m][s] stage-cost words; X: [L+1][C] link costs.
    """
    L, Du, unit, C, Pmax, M = inst.L, inst.D // inst.unit, inst.unit, len(inst.cand), inst.Pmax, inst.M
    G = [int(g) for g in inst.tierG]
    cand = [int(c) for c in inst.cand]
    K = 0
    while (1 << K) <= Du:
        K += 1

    def pair(i, j):
        return i * L - i * (i - 1) // 2 + (j - i - 1)

    for P in range(1, min(Pmax, L) + 1):
        for cuts in itertools.combinations(range(1, L), P - 1):
            bounds = (0,) + cuts + (L,)
            for ms in itertools.product(range(K), repeat=P):
                if sum(1 << m for m in ms) > Du:
                    continue
                for cs in itertools.product(range(C), repeat=P - 1):
                    ok = True
                    bott = 0
                    for q in range(P):
                        i, j, m = bounds[q], bounds[q + 1], ms[q]
                        k = unit << m
                        pos = P - q
                        if q > 0 and 2 * k > G[cand[cs[q - 1]]]:
                            ok = False
                            break
                        if q < P - 1 and 2 * k > G[cand[cs[q]]]:
                            ok = False
                            break
                        tau = stage_min_tau(words[pair(i, j)][m], pos)
                        if tau is None:
                            ok = False
                            break
                        cost = tau
                        if q > 0:
                            cost += int(X[i][cs[q - 1]])
                        if q < P - 1:
                            cost += int(X[j][cs[q]])
                        bott = max(bott, cost)
                    if not ok or bott >= CAP:
                        continue
                    yield bott * (M + P - 1), P, bott, (bounds, ms, cs)


def brute_optimum(inst, words, X):
    """(t_batch, P, bottleneck) of the best plan, ties to fewer stages; None if none."""
    best = None
    for t, P, v, _ in enumerate_plans(inst, words, X):
        if best is None or (t, P) < (best[0], best[1]):
            best = (t, P, v)
    return best


def price_plan(inst, words, X, plan):
    """Price a plan given as [(i, j, k, s, c_next)]: returns (t_batch, bottleneck)
    or None when a stage is infeasible at its position or breaks a width rule."""
    L = inst.L
    G = [int(g) for g in inst.tierG]
    cand = [int(c) for c in inst.cand]
    P = len(plan)

    def pair(i, j):
        return i * L - i * (i - 1) // 2 + (j - i - 1)

    bott = 0
    prev_c = None
    used = 0
    for q, (i, j, k, s, cn) in enumerate(plan):
        m = (k // inst.unit).bit_length() - 1
        used += k // inst.unit
        w = int(words[pair(i, j)][m][s])
        if w == INF or (w & 0xFF) < P - q:
            return None
        cost = w >> 8
        if q > 0:
            if 2 * k > G[cand[prev_c]]:
                return None
            cost += int(X[i][prev_c])
        if q < P - 1:
            if cn < 0 or 2 * k > G[cand[cn]]:
                return None
            cost += int(X[j][cn])
        bott = max(bott, cost)
        prev_c = cn
    if used > inst.D // inst.unit or plan[0][0] != 0 or plan[-1][1] != L:
        return None
    return bott * (inst.M + P - 1), bott
