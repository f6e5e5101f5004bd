"""Host-side check of the cost builder's exact division by invariant divisors
(Granlund & Montgomery 1994, Fig. 4.1) against the C++ division operator."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_invariant_divisor_matches_division(tmp_path):
    exe = tmp_path / "divisor_check"
    subprocess.check_call(["g++", "-O2", "-std=c++17", os.path.join(HERE, "native", "divisor_check.cpp"),
                           "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert " 0 wrong" in out.stdout
