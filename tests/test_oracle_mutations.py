"""The oracle's pins catch plausible mistakes (CPU only).

For every entry of ``oracle_mutations.MUTATIONS`` -- one slip planted in one
oracle expression -- the named pin files run in a child pytest with the slip
in place, and at least one pin must fail.  A slip no pin notices would mean
the oracle is pinned only to itself there.
"""

import os
import subprocess
import sys

import pytest

from oracle_mutations import MUTATIONS

TESTS = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name):
    files = MUTATIONS[name][3]
    env = dict(os.environ, QMUON_PLANT_ORACLE_MISTAKE=name)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        *files], cwd=TESTS, env=env, capture_output=True, text=True, timeout=600)
    # exit status 1: tests ran and at least one failed (not a crash or a planting error)
    assert r.returncode == 1 and " failed" in r.stdout, (name, r.returncode, r.stdout[-1500:], r.stderr[-1500:])
