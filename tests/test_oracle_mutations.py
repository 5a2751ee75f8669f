"""A sample of the oracle mutation check inside the CPU suite.

tests/oracle_mutations.py plants each of its mistakes in a temporary copy of the oracle and
requires a pin to fail.  The full list takes a few minutes; here one mistake per part of the
oracle runs on every suite run, so a pin weakened later is noticed.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))

SAMPLE = ["q2k unpack shift", "q2k nibbles swapped", "half normal bias", "q2k enc min unclamped",
          "q4k unpack sc hi", "q4k enc d /62", "route ties to higher index", "group perm holds tokens",
          "routed swiglu operands", "shared down transposed", "expert blob gate and up swapped",
          "steer dot operand"]


def test_sampled_mutations_are_caught():
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_mutations.py"), *SAMPLE],
                       capture_output=True, text=True, timeout=900)
    lines = [l for l in r.stdout.splitlines() if ": " in l and "|" in l]
    assert len(lines) == len(SAMPLE), r.stdout + r.stderr
    assert r.returncode == 0, r.stdout
