"""Register and spill budgets of the kernels, from ptxas's resource report
(CPU only: nvcc cross-compiles for sm_103a without a GPU).

The update kernel runs 3 CTAs of 288 threads per SM, so it has at most 72
registers a thread; the Newton-Schulz kernel runs one CTA of 10 warps per SM
and is capped at 168.  A spill in their hot loops cost the update kernel a
quarter of its bandwidth once, so the kernels that carry the bf16 and fp16
paths, the Newton-Schulz products and the GRASP passes must not spill at
all.  (The fp32-gradient update variants spill a little today; they are not
on the benchmarked path.)
"""

import os
import re
import shutil
import subprocess

import pytest

from memory_reduced_muon_gb300 import build

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def _report(src, tmp_path):
    out = tmp_path / (os.path.basename(src) + ".o")
    r = subprocess.run([build.nvcc(), *build.ARCH, *build.FLAGS, "-Xptxas", "-v", "-c", src, "-o", str(out)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    kernels, cur = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            kernels[cur] = {}
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur:
            kernels[cur]["spill"] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            kernels[cur]["regs"] = int(m.group(1))
    assert kernels
    return kernels


def test_update_kernels_fit_three_ctas_without_spills(tmp_path):
    k = _report(os.path.join(build.CSRC, "update.cu"), tmp_path)
    upd = {n: v for n, v in k.items() if "update_kernel" in n}
    assert len(upd) == 18                        # q8 kind x grad dtype x (plain, carrier, stochastic)
    for name, v in upd.items():
        assert v["regs"] <= 72, (name, v)
        dt = int(re.search(r"update_kernelILi\dELi(\d)E", name).group(1))
        if dt != 2:                              # bf16 and fp16 gradients
            assert v["spill"] == 0, (name, v)


# Spills accepted as they stand in the measured kernels: none.  Any growth
# fails.
SPILL_BUDGET = {}


def test_newton_schulz_and_grasp_kernels_do_not_spill(tmp_path):
    for src, cap in (("ns_gemm.cu", 168), ("grasp.cu", 255)):
        k = _report(os.path.join(build.CSRC, src), tmp_path)
        for name, v in k.items():
            budget = next((b for key, b in SPILL_BUDGET.items() if key in name), 0)
            assert v["spill"] <= budget, (src, name, v)
            assert v["regs"] <= cap, (src, name, v)
