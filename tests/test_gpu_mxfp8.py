"""GPU parity of the MXFP8 carrier path: update -> carrier -> Newton-Schulz.

The carrier (E4M3 payload, E8M0 scale per 32 row elements, fp32 inverse
norm) feeds ``qmuon_newton_schulz_batched`` directly.  Checks: the result is
bit-identical to the bf16 path run on the oracle's exact decode of the same
carrier (so the expansion is exact), and it is within the MXFP8 tolerance
(relative Frobenius 5e-2, per-row cosine 0.995) of the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import carrier, ns

from gpu_util import bf16_to_f64, min_row_cos, rel_fro, to_oracle_grad

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(256, 1024), (1024, 256), (96, 160), (512, 512)])
def test_carrier_to_newton_schulz(shape):
    rows, cols = shape
    w = workloads.get(5)
    m = workloads.Matrix("t", rows, cols)
    g = workloads.make_grad(w, 0, 1, device="cuda", matrix=m)
    qs, a = workloads.zero_state(m, "int8", device="cuda")
    hq, ha, hg = qs.cpu().numpy(), a.cpu().numpy(), to_oracle_grad(g, "bf16")
    payload = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows * (cols // 32), dtype=torch.uint8, device="cuda")
    inv = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_carrier_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier(qs, a, g, rows, cols, "int8", "bf16", w.beta, payload, scale, inv, ws)
    r = carrier.carrier_update(hq, ha, hg, w.beta, rows, cols)
    np.testing.assert_array_equal(payload.cpu().numpy().reshape(rows, cols), r.payload)

    out = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    prob = q.ns_problem(out, rows, cols, inv_norm=inv, input_kind=q.QMUON_NS_MXFP8, payload=payload,
                        scale_inv=scale)
    ws2 = torch.empty(q.qmuon_ns_workspace_size([prob]), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched([prob], 5, w.coeffs, ws2)
    q.qmuon_sync_status(ws2)

    # the bf16 path on the oracle's decode of the same carrier
    dec = carrier.decode_rows(r.payload, r.scale_inv)          # fp64, exact
    x16 = torch.from_numpy(dec.astype(np.float32)).to(torch.bfloat16).cuda()
    assert np.array_equal(x16.float().cpu().numpy().astype(np.float64), dec)   # exact in bf16
    q.qmuon_newton_schulz_batched([q.ns_problem(x16, rows, cols, inv_norm=inv)], 5, w.coeffs, ws2)
    q.qmuon_sync_status(ws2)
    assert torch.equal(out.view(torch.int16), x16.view(torch.int16))

    ref = ns.newton_schulz(dec, inv_norm=float(inv.item()))
    got = bf16_to_f64(out)
    assert rel_fro(got, ref) <= 5e-2 and min_row_cos(got, ref) >= 0.995
    # the carrier's inverse norm is the update's
    np.testing.assert_allclose(inv.item(), r.inv_norm, rtol=1e-5)
