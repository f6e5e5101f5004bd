"""The benchmark's work counts against a direct loop over the recurrence's transitions.

A relaxation is one (j, m, c') min-max transition of Eq. 3 (Nest §4) for one DP cell
(i, d, p, c) whose successor cell dp[j][d - 2^m][p - 1][c'] can hold a value (state j
keeps at least p - 1 layers and d - 2^m >= p - 1 device units remain for the p - 1
stages after the new one); with the strategy axis it is one (j, m, s, c') transition.
The bench counts them with vectorised sums; here every cell and transition is
enumerated.
"""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from memory_aware_device_gb300 import synth  # noqa: E402


def direct(x, with_strategies):
    Du, P, C, u = x.D // x.unit, x.Pmax, len(x.cand), x.unit
    G = [int(x.tierG[c]) for c in x.cand]
    st = bench.states(x)
    E = len(st) - 1
    moe = sum(1 << l for l in range(x.L) if int(x.moe[l]))
    n = 0
    for i in range(E):
        for d in range(1, Du + 1):
            for p in range(1, min(P, bin(st[i]).count("1")) + 1):
                for c in range(1 if i == 0 else C):
                    for j in range(i + 1, E + 1):
                        if st[j] & ~st[i] or (j == E) != (p == 1):
                            continue
                        if bin(st[j]).count("1") < p - 1:   # too few layers left for p - 1 stages
                            continue
                        for m in range(Du.bit_length()):
                            k = u << m
                            if (1 << m) > d - (p - 1) or (i > 0 and 2 * k > G[c]):
                                continue
                            ns = 1
                            if with_strategies:
                                hm = bool((st[i] & ~st[j]) & moe)
                                ns = sum(1 for t, cp, e, _, _ in x.strat
                                         if not (k % (int(t) * int(cp)) or (k // (int(t) * int(cp))) % int(e)
                                                 or (int(e) > 1 and not hm)))
                            ncp = 1 if j == E else sum(1 for g in G if 2 * k <= g)
                            n += ns * ncp
    return n


@pytest.mark.parametrize("seed", range(30))
def test_counts_match_a_direct_loop(seed):
    x = synth.random_tiny(seed + 500, Lmax=6, Dmax=8)
    if seed % 2:
        x.succ = synth.random_dag(seed, x.L, (0.2, 0.5)[seed % 4 // 2])
    assert bench.relaxations(x) == direct(x, False)
    assert bench.relaxations_with_strategies(x) == direct(x, True)


def test_workload_counts():
    # the (j, k, c') and (j, k, s, c') counts of the dense 32-layer workload (16 instances)
    # and of the tiny 8-layer one, as the work-per-batch sizing gives them
    batch = synth.config_batch(2)
    assert sum(bench.relaxations(x) for x in batch) == 57229968
    assert sum(bench.relaxations_with_strategies(x) for x in batch) == 394430160
    tiny = synth.config_instance(1, 0)
    assert (bench.relaxations(tiny), bench.relaxations_with_strategies(tiny)) == (1216, 4326)
    x = synth.two_tower_instance(0)
    assert bench.relaxations(x) == direct(x, False)
    assert bench.state_pairs(x) == 96 * 97 // 2


def test_relax_peak_mode():
    # the roofline divides by the peak of the words the sweep runs on
    resident, streaming = {"sweep_variant": 1}, {"sweep_variant": 2}
    dense = synth.config_batch(2, B=2)                       # two candidates: tagged words
    torus = [synth.torus_instance(b) for b in range(2)]      # three candidates: plain words
    assert len(dense[0].cand) == 2 and len(torus[0].cand) == 3
    assert bench.relax_peak_mode(dense, resident) == 2
    assert bench.relax_peak_mode(torus, resident) == 0
    assert bench.relax_peak_mode(dense, streaming) == 1
    assert bench.relax_peak_mode(dense + torus, resident) == 0


def test_reference_arm_line():
    # the reference arm (the oracle on the host cores) prints one JSON line with the
    # GPU arm's metric, unit and config, and no host-device traffic
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "2", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"]) == (bench.METRIC, bench.UNIT)
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (3, 3, 1)
    batch = synth.config_batch(2)
    words = sum(bench.cost_words(x) for x in batch)
    assert line["config"] == bench.bench_config("dense-32L-h4096-64dev", batch, len(batch),
                                                57229968, words, 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT,
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # under torchrun only rank 0 runs it; the other ranks exit 0 without output
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "2", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=root, env=env)
    assert out.returncode == 0 and out.stdout.strip() == "", (out.stdout, out.stderr[-2000:])
