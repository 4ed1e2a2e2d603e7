"""The oracle's pins catch plausible mistakes in the oracle itself.

Each mutant of tests/oracle_mutants.py plants one mistake in the fp64 oracle (on the CPU, in a
child process): a rotation turning the wrong way, theta indexed from 1, the diagonal masked, a
window one key too wide, the split-halves pairing ignored, softmax over the wrong axis, the
log-sum-exp in log2 units, values of the wrong key, 1/D instead of 1/sqrt(D), the wrong K/V head
for a query head, the decode query rotated one position too far, the rotary part dropped from the
absorbed MLA query, and the wrong head's W_UV.  The pins (tests/test_oracle.py,
tests/test_workloads.py) must fail under every one of them, and pass without any.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from tests.oracle_mutants import MUTANTS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle.py", "tests/test_workloads.py"]


def run_pins(mutant: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, ORACLE_MUTANT=mutant)
    cmd = [sys.executable, "-m", "pytest", *PINS, "-q", "-x", "-p", "tests.oracle_mutants", "-p", "no:cacheprovider"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def results():
    names = [""] + sorted(MUTANTS)
    with cf.ThreadPoolExecutor(max_workers=min(8, len(names))) as ex:
        return dict(zip(names, ex.map(run_pins, names)))


def test_pins_pass_without_a_mutant(results):
    r = results[""]
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(results, mutant):
    r = results[mutant]
    # exit code 1: some test failed (not a collection or usage error, which would be 2 or more)
    assert r.returncode == 1, f"mutant {mutant} survived the pins (exit {r.returncode}):\n{r.stdout[-2000:]}"
