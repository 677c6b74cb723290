"""CPU oracle for the quantized Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA library in ``memory_reduced_muon_gb300`` and the
library never falls back to it.

What it computes, and where that is defined:

* ``oracle.codec``   -- the blockwise 8-bit momentum codec and update, the
  grouped sum-of-squares and the inverse Frobenius norms
  ("Quantized Muon Momentum", sections "Algorithm" and "Grouped QKV And
  Sharding").  fp32 arithmetic in the stated operation order, fp64 sums.
* ``oracle.carrier`` -- the MXFP8 carrier (E4M3 payload, E8M0 scale per 32
  row elements, fp32 inverse norm) ("Quantized Muon Momentum", section
  "Wave18B MXFP8 Carrier Probe").
* ``oracle.ns``      -- quintic Newton-Schulz orthogonalisation in fp64
  ("NVIDIA impulsa optimizadores avanzados ... con Megatron", section
  "Newton-Schulz distribuido": three matrix products per iteration).
* ``oracle.muonbp``  -- the MuonBP block-periodic step with two learning
  rates ("MuonBP: Faster Muon via Block-Periodic Orthogonalization",
  section "整体框架", flowchart, and "关键设计" items 1-3).
* ``oracle.rng``     -- the Philox4x32-10 counter-based generator (Salmon et
  al., SC'11) that draws the offsets of the stochastic requantisation in
  ``oracle.codec`` (a reading: the momentum page lists stochastic rounding
  as not yet implemented, section "Known Limitations").
* ``oracle.grasp``   -- the 4-bit GRASP momentum state: a rank-8 factor
  refreshed by one warm-started power iteration plus a grid-quantised
  residual ("4-bit-Muon-GRASP", the update equations and the grid
  quantisation on that page).

Every function names the passage it follows.  Where the pages are silent the
docstring states the reading taken.  Pins (tests that tie each function to
something other than itself) live in ``tests/test_oracle_*.py``; a function
without one would say "parity unpinned" here -- at present every function is
pinned.
"""

from . import codec, carrier, ns, muonbp  # noqa: F401
