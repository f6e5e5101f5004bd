"""Writes workload5_results.txt: the CPU oracle's results for every instance of the
mixed-128L-4096dev-stress workload (128 alternating dense / MoE layers, hidden
4096 / 8192 / 16384, 4096 devices in four tiers, 672 strategies, 1024 instances).

Each line holds the instance index, a fingerprint of its inputs (so that a change of
the input generator shows as a clear mismatch instead of a parity failure), and what
the oracle returns for it: status, t_batch, the bottleneck stage time and the plan,
each stage as i:j:k:s:c_next (Nest §4 Eq. 3 solved backward, then Appendix K
Algorithm 1's batch-time loop and stage reconstruction).

Only the oracle computes these values; the script runs the instances on a thread
pool (each instance single-threaded; the oracle's C calls release the GIL):

    python tests/golden/make_workload5_results.py [--threads N]
"""
from __future__ import annotations

import argparse
import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from memory_aware_device_gb300 import synth  # noqa: E402
from oracle import oracle as O  # noqa: E402

OUT = os.path.join(HERE, "workload5_results.txt")
WORKLOAD = 5


def fingerprint(x) -> str:
    """16 hex digits of SHA-256 over an instance's scalars and input arrays."""
    h = hashlib.sha256()
    h.update(np.asarray([x.L, x.D, x.unit, x.Pmax, x.R, x.M, x.budget, x.opt_factor, x.schedule],
                        dtype=np.int64).tobytes())
    for a, dt in ((x.fl, np.int64), (x.pd, np.int64), (x.pe, np.int64), (x.ao, np.int64),
                  (x.aw, np.int64), (x.a2a, np.int64), (x.moe, np.uint8), (x.tierG, np.int64),
                  (x.tierBw, np.int64), (x.tierLat, np.int64), (x.cand, np.int32), (x.strat, np.int16)):
        h.update(np.ascontiguousarray(np.asarray(a, dtype=dt)).tobytes())
    return h.hexdigest()[:16]


def format_line(b: int, fp: str, r: dict) -> str:
    stages = " ".join(f"{i}:{j}:{k}:{s}:{c}" for i, j, k, s, c in r["plan"])
    return f"{b} {fp} {r['status']} {r['t_batch']} {r['bottleneck']} {len(r['plan'])}" + (f" {stages}" if stages else "")


def parse(path: str = OUT) -> dict:
    """{b: (fingerprint, status, t_batch, bottleneck, plan)} from a results file."""
    out = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        b, fp, st, t, v, n = int(f[0]), f[1], int(f[2]), int(f[3]), int(f[4]), int(f[5])
        plan = [tuple(int(q) for q in s.split(":")) for s in f[6:6 + n]]
        out[b] = (fp, st, t, v, plan)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    args = ap.parse_args()
    from concurrent.futures import ThreadPoolExecutor
    B = synth.CONFIG_BATCH[WORKLOAD]
    O.lib()
    t0 = time.time()

    def one(b):
        x = synth.config_instance(WORKLOAD, b)
        return b, fingerprint(x), O.solve(x)

    lines = [None] * B
    with ThreadPoolExecutor(max_workers=args.threads) as ex:
        for n, (b, fp, r) in enumerate(ex.map(one, range(B)), 1):
            lines[b] = format_line(b, fp, r)
            if n % 64 == 0:
                print(f"{n}/{B} instances, {time.time() - t0:.0f} s", flush=True)
    with open(OUT + ".tmp", "w") as f:
        f.write(f"# CPU oracle results, {synth.CONFIG_NAMES[WORKLOAD]}, {B} instances "
                f"(seed 1000*{WORKLOAD} + b); written by make_workload5_results.py\n")
        f.write("# b input_fingerprint status t_batch bottleneck n_stages i:j:k:s:c_next ...\n")
        for line in lines:
            f.write(line + "\n")
    os.replace(OUT + ".tmp", OUT)
    print(f"wrote {OUT} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
