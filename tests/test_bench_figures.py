"""The DRAM-traffic figures bench.py reports beside its rates come from the
committed ncu summaries under profiles/ (``key = bytes`` lines).  Each key the
bench reads must be there, with a value of the size a full-size launch or call
moves, so that an edit of a summary cannot silently turn a reported traffic
figure into null.  CPU only."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_bench_finds_every_traffic_figure():
    t = bench.load_traffic()
    # (key, algorithmic bytes of the full-size launch or call it stands for)
    expected = {
        "update_bytes_per_launch": 6.031 * 872415232,      # the momentum update, 4 Llama-8B layers
        "update_sr_bytes_per_launch": 6.031 * 872415232,   # the same with stochastic requantisation
        "grasp_bytes_per_call": 9.25 * 872415232,          # one GRASP call on the same matrices
        "ns_block_bytes_per_call": None,                   # one Newton-Schulz call on the block set
    }
    for key, alg in expected.items():
        assert key in t, key
        assert t[key] > 1e9, (key, t[key])
        if alg is not None:
            # measured DRAM bytes within 10% of the algorithmic bytes: no re-reads,
            # a few dirty lines still in L2 at the end
            assert 0.9 * alg <= t[key] <= 1.1 * alg, (key, t[key], alg)
