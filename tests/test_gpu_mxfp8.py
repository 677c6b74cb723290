"""GPU parity of the MXFP8 carrier path: update -> carrier -> Newton-Schulz.

The carrier (E4M3 payload, E8M0 scale per 32 row elements, fp32 inverse
norm) feeds ``qmuon_newton_schulz_batched`` directly; the engine expands it
exactly (an E4M3 value times a power of two fits in bf16) and runs its bf16
tensor-core products on it.  Checks:
- one iteration with only the b A term on: within the single-product
  tolerance (6e-3) of fp64 products of the oracle's exact decode at the
  engine's bf16 rounding points, on shapes with ragged 128-row blocks,
  partial 128-column groups and several SYRK tiles (mirrored ones included);
- five iterations: bit-identical to the bf16 path run on the oracle's exact
  decode of the same carrier, and within the MXFP8 tolerance (relative
  Frobenius 5e-2, per-row cosine 0.995) of the fp64 oracle, wide and tall;
- a batch mixing carriers and a bf16 problem.
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import carrier, ns

from gpu_util import bf16_to_f64, min_row_cos, one_iteration_reference, rel_fro, to_oracle_grad

pytestmark = pytest.mark.gpu


def _carrier(rows, cols, seed_step=1):
    """A carrier from one update of a zero state (grad of the carrier
    workload's distribution), on the GPU and in the oracle."""
    w = workloads.get(5)
    m = workloads.Matrix("t", rows, cols)
    g = workloads.make_grad(w, 0, seed_step, device="cuda", matrix=m)
    qs, a = workloads.zero_state(m, "int8", device="cuda")
    hq, ha, hg = qs.cpu().numpy(), a.cpu().numpy(), to_oracle_grad(g, "bf16")
    payload = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows * (cols // 32), dtype=torch.uint8, device="cuda")
    inv = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_carrier_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier(qs, a, g, rows, cols, "int8", "bf16", w.beta, payload, scale, inv, ws)
    r = carrier.carrier_update(hq, ha, hg, w.beta, rows, cols)
    np.testing.assert_array_equal(payload.cpu().numpy().reshape(rows, cols), r.payload)
    np.testing.assert_array_equal(scale.cpu().numpy().reshape(rows, cols // 32), r.scale_inv)
    return payload, scale, inv, r


def _ns_from_carrier(payload, scale, inv, rows, cols, iters, coeffs):
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    prob = q.ns_problem(out, rows, cols, inv_norm=inv, input_kind=q.QMUON_NS_MXFP8, payload=payload,
                        scale_inv=scale)
    ws = torch.empty(q.qmuon_ns_workspace_size([prob]), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched([prob], iters, coeffs, ws)
    q.qmuon_sync_status(ws)
    return out


# Ragged 128-row blocks (96, 300), a partial 128-column group (160, 1312),
# several SYRK tiles with mirrored ones (640 rows), a tall carrier.
MX_SHAPES = [(256, 1024), (96, 160), (512, 512), (300, 544), (640, 1312), (128, 4096), (1312, 640)]


@pytest.mark.parametrize("shape", MX_SHAPES)
def test_carrier_gram_single_product(shape):
    rows, cols = shape
    payload, scale, inv, r = _carrier(rows, cols)
    coeffs = (0.0, 1.0, 0.0)   # X1 = inv * bf16(b A) X0 with A = bf16(inv^2 X0 X0^T)
    out = _ns_from_carrier(payload, scale, inv, rows, cols, 1, coeffs)
    dec = carrier.decode_rows(r.payload, r.scale_inv)          # fp64, exact
    ref = one_iteration_reference(dec, coeffs, float(inv.item()))
    err = rel_fro(bf16_to_f64(out), ref)
    assert err <= 6e-3, (shape, err)


@pytest.mark.parametrize("shape", [(256, 1024), (1024, 256), (96, 160), (512, 512), (640, 1312), (1312, 640)])
def test_carrier_to_newton_schulz(shape):
    rows, cols = shape
    w = workloads.get(5)
    payload, scale, inv, r = _carrier(rows, cols)
    out = _ns_from_carrier(payload, scale, inv, rows, cols, 5, w.coeffs)
    dec = carrier.decode_rows(r.payload, r.scale_inv)          # fp64, exact
    ref = ns.newton_schulz(dec, inv_norm=float(inv.item()))
    got = bf16_to_f64(out)
    assert rel_fro(got, ref) <= 5e-2 and min_row_cos(got, ref) >= 0.995, (shape, rel_fro(got, ref))

    # the bf16 path on the oracle's decode of the same carrier
    x16 = torch.from_numpy(dec.astype(np.float32)).to(torch.bfloat16).cuda()
    assert np.array_equal(x16.float().cpu().numpy().astype(np.float64), dec)   # exact in bf16
    ws2 = torch.empty(q.qmuon_ns_workspace_size([q.ns_problem(x16, rows, cols)]), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched([q.ns_problem(x16, rows, cols, inv_norm=inv)], 5, w.coeffs, ws2)
    q.qmuon_sync_status(ws2)
    got16 = bf16_to_f64(x16)
    assert rel_fro(got16, ref) <= 5e-2 and min_row_cos(got16, ref) >= 0.995
    # the carrier is expanded exactly: the same bits as the bf16 path
    assert torch.equal(out.view(torch.int16), x16.view(torch.int16))
    # the carrier's inverse norm is the update's
    np.testing.assert_allclose(inv.item(), r.inv_norm, rtol=1e-5)


def test_mixed_batch_carrier_and_bf16():
    # a batch holding a wide carrier, a tall carrier and a bf16 problem
    w = workloads.get(5)
    p1, s1, i1, r1 = _carrier(256, 1024)
    p2, s2, i2, r2 = _carrier(640, 256, seed_step=2)
    rng = np.random.default_rng(3)
    M3 = torch.from_numpy(rng.standard_normal((384, 512)).astype(np.float32)).to(torch.bfloat16).cuda()
    M3_in = bf16_to_f64(M3)
    inv3 = torch.tensor([1.0 / np.linalg.norm(M3_in)], dtype=torch.float32, device="cuda")
    o1 = torch.empty(256, 1024, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty(640, 256, dtype=torch.bfloat16, device="cuda")
    probs = [q.ns_problem(o1, 256, 1024, inv_norm=i1, input_kind=q.QMUON_NS_MXFP8, payload=p1, scale_inv=s1),
             q.ns_problem(o2, 640, 256, inv_norm=i2, input_kind=q.QMUON_NS_MXFP8, payload=p2, scale_inv=s2),
             q.ns_problem(M3, 384, 512, inv_norm=inv3)]
    ws = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, 5, w.coeffs, ws)
    q.qmuon_sync_status(ws)
    for out, r, inv in ((o1, r1, i1), (o2, r2, i2)):
        ref = ns.newton_schulz(carrier.decode_rows(r.payload, r.scale_inv), inv_norm=float(inv.item()))
        got = bf16_to_f64(out)
        assert rel_fro(got, ref) <= 5e-2 and min_row_cos(got, ref) >= 0.995
    ref3 = ns.newton_schulz(M3_in, inv_norm=float(inv3.item()))
    got3 = bf16_to_f64(M3)
    assert rel_fro(got3, ref3) <= 2e-2 and min_row_cos(got3, ref3) >= 0.999
