"""The oracle's pins catch plausible mistakes (CPU only).

For every entry of ``oracle_mutations.MUTATIONS`` -- one slip planted in one
oracle expression -- the named pin files run in a child pytest with the slip
in place, and at least one pin must fail.  A slip no pin notices would mean
the oracle is pinned only to itself there.  The children run in parallel.
"""

import concurrent.futures as cf
import os
import subprocess
import sys

from oracle_mutations import MUTATIONS

TESTS = os.path.dirname(os.path.abspath(__file__))


def _run(name):
    files = MUTATIONS[name][3]
    env = dict(os.environ, QMUON_PLANT_ORACLE_MISTAKE=name)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        *files], cwd=TESTS, env=env, capture_output=True, text=True, timeout=600)
    # exit status 1: tests ran and at least one failed (not a crash or a planting error)
    caught = r.returncode == 1 and " failed" in r.stdout
    return name, caught, f"exit {r.returncode}: {r.stdout[-400:]} {r.stderr[-400:]}"


def test_every_planted_mistake_fails_a_pin():
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(_run, sorted(MUTATIONS)))
    missed = [(name, detail) for name, caught, detail in results if not caught]
    assert not missed, missed
