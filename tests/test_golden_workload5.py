"""The stored oracle results of the mixed-128L workload (tests/golden/workload5_results.txt)
still describe what the generator draws and what the oracle computes: every input
fingerprint matches, and re-solving a few instances with the oracle reproduces their
lines.  The GPU parity test compares all 1024 GPU results with this file."""
import importlib.util
import os

from memory_aware_device_gb300 import synth
from oracle import oracle as O

HERE = os.path.join(os.path.dirname(__file__), "golden")


def _mod():
    spec = importlib.util.spec_from_file_location("make_workload5_results",
                                                  os.path.join(HERE, "make_workload5_results.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_fingerprint_matches_the_generator():
    mod = _mod()
    gold = mod.parse()
    assert sorted(gold) == list(range(synth.CONFIG_BATCH[5]))
    for b in range(0, 1024, 97):
        assert gold[b][0] == mod.fingerprint(synth.config_instance(5, b)), b


def test_oracle_reproduces_stored_lines():
    mod = _mod()
    gold = mod.parse()
    for b in (3, 700):
        x = synth.config_instance(5, b)
        r = O.solve(x)
        fp, st, t, v, plan = gold[b]
        assert (r["status"], r["t_batch"], r["bottleneck"], r["plan"]) == (st, t, v, plan), b
