"""The path and dtype audit (qmuon_get_counters) on the GPU: every entry that
computes adds what it enqueued, by path and dtype, and nothing else.

The page's carrier probe ("Quantized Muon Momentum", §Wave18B MXFP8 Carrier
Probe) audits a run by counting carrier-update calls and the dtypes of the
tensors involved (uint8 payload and scales, fp32 inverse norm, the gradient's
dtype).  Here one test drives every computing entry once, with small shapes,
and checks each tally against the calls it made; the bf16 hand-off of a
carrier batch is checked as 2 bytes per carrier element.
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import grasp

pytestmark = pytest.mark.gpu

COEFFS = workloads.COEFFS


def _grad(rows, cols, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(rows, cols, generator=g, device="cuda") * 1e-2).to(dtype).contiguous()


def _state(rows, cols, kind="int8"):
    return workloads.zero_state(workloads.Matrix("t", rows, cols), kind, device="cuda")


def _delta(before, after):
    return {k: after[k] - before[k] for k in after}


def _expect(delta, **want):
    # every field not named must be unchanged
    full = {k: 0 for k in q.COUNTER_FIELDS}
    full.update(want)
    assert delta == full, {k: (delta[k], full[k]) for k in full if delta[k] != full[k]}


def test_counters_follow_every_path():
    torch.cuda.synchronize()
    shapes = [(256, 512), (128, 1024)]

    # ---- planned update, nearest and stochastic ----
    states = [_state(r, c) for r, c in shapes]
    grads = [_grad(r, c, 10 + i) for i, (r, c) in enumerate(shapes)]
    plan = q.qmuon_plan_create([(s[0], s[1], g, r, c) for s, g, (r, c) in zip(states, grads, shapes)],
                               "int8", "bf16")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    inv = torch.zeros(len(shapes), device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_update_multi_normalize_groups(plan, 0.95, 2, None, inv, ws)
    _expect(_delta(c0, q.qmuon_get_counters()), update_calls=1, grad_bf16_tensors=2, state_int8_tensors=2)
    c0 = q.qmuon_get_counters()
    q.qmuon_update_multi_normalize_groups_sr(plan, 0.95, 2, 7, 1, None, inv, ws)
    _expect(_delta(c0, q.qmuon_get_counters()), update_calls=1, update_sr_calls=1, grad_bf16_tensors=2,
            state_int8_tensors=2)
    q.qmuon_sync_status(ws)

    # ---- the allocation-free update: fp16 gradient, uint8 state ----
    sq, sa = _state(64, 256, "uint8")
    g16 = _grad(64, 256, 3, torch.float16)
    c0 = q.qmuon_get_counters()
    q.qmuon_update_normalize_noalloc(sq, sa, g16, 64, 256, "uint8", "f16", 0.9)
    q.qmuon_noalloc_sync_status()
    _expect(_delta(c0, q.qmuon_get_counters()), update_calls=1, grad_fp16_tensors=1, state_uint8_tensors=1)

    # ---- carriers: one tensor (fp32 gradient), then a plan's worth ----
    rows, cols = 96, 160
    cq, ca = _state(rows, cols)
    g32 = _grad(rows, cols, 4, torch.float32)
    payload = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows * (cols // 32), dtype=torch.uint8, device="cuda")
    cinv = torch.zeros(1, device="cuda")
    cws = torch.empty(q.qmuon_carrier_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_update_mxfp8_carrier(cq, ca, g32, rows, cols, "int8", "f32", 0.9, payload, scale, cinv, cws)
    _expect(_delta(c0, q.qmuon_get_counters()), carrier_calls=1, grad_fp32_tensors=1, state_int8_tensors=1,
            carrier_payload_u8_tensors=1, carrier_scale_u8_tensors=1, carrier_inv_norm_f32_values=1)
    payloads = [torch.empty(r * c, dtype=torch.uint8, device="cuda") for r, c in shapes]
    scales = [torch.empty(r * (c // 32), dtype=torch.uint8, device="cuda") for r, c in shapes]
    invs = torch.zeros(len(shapes), device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_update_mxfp8_carrier_multi(plan, 0.9, payloads, scales, invs, ws)
    _expect(_delta(c0, q.qmuon_get_counters()), carrier_calls=1, grad_bf16_tensors=2, state_int8_tensors=2,
            carrier_payload_u8_tensors=2, carrier_scale_u8_tensors=2, carrier_inv_norm_f32_values=2)
    q.qmuon_sync_status(ws)

    # ---- Newton-Schulz on a batch of two carriers and one bf16 problem ----
    outs = [torch.empty(r, c, dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    probs = [q.ns_problem(o, r, c, inv_norm=invs[i:i + 1], input_kind=q.QMUON_NS_MXFP8, payload=payloads[i],
                          scale_inv=scales[i]) for i, (o, (r, c)) in enumerate(zip(outs, shapes))]
    xb = _grad(512, 256, 5)
    probs.append(q.ns_problem(xb, 512, 256, inv_norm=inv[0:1]))
    nws = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_newton_schulz_batched(probs, 5, COEFFS, nws)
    _expect(_delta(c0, q.qmuon_get_counters()), ns_calls=1, ns_mxfp8_problems=2, ns_bf16_problems=1,
            ns_bf16_handoff_bytes=2 * sum(r * c for r, c in shapes))
    q.qmuon_sync_status(nws)

    # ---- steps: a block step on a 1 x 2 tiling, a full step, a host-fed one, stochastic ----
    splan = q.qmuon_plan_create([(s[0], s[1], g, r, c) for s, g, (r, c) in zip(states, grads, shapes)],
                                "int8", "bf16", tile=(1, 2))
    sws = torch.empty(q.qmuon_workspace_size(splan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    weights = [torch.zeros(r, c, device="cuda") for r, c in shapes]
    sums = torch.zeros(len(shapes) * 2, device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_step(splan, 1, 2, 0.95, 0.02, 0.01, weights, COEFFS, 5, sums, sws)
    _expect(_delta(c0, q.qmuon_get_counters()), step_block_calls=1, grad_bf16_tensors=2, state_int8_tensors=2,
            ns_bf16_problems=4, weight_f32_tensors=2)
    c0 = q.qmuon_get_counters()
    q.qmuon_step(splan, 2, 2, 0.95, 0.02, 0.01, weights, COEFFS, 5, sums, sws)
    _expect(_delta(c0, q.qmuon_get_counters()), step_full_calls=1, grad_bf16_tensors=2, state_int8_tensors=2,
            ns_bf16_problems=2, weight_f32_tensors=2)
    host = [_grad(r, c, 20 + i).cpu().pin_memory() for i, (r, c) in enumerate(shapes)]
    hsum = torch.zeros(len(shapes) * 2).pin_memory()
    q.qmuon_plan_set_stochastic_rounding(splan, True, 11)
    c0 = q.qmuon_get_counters()
    q.qmuon_step_from_host(splan, 3, 2, 0.95, 0.02, 0.01, weights, COEFFS, 5, host, hsum, sums, sws)
    # torch's page-locked buffers are mapped: the step reads them with its own loads
    _expect(_delta(c0, q.qmuon_get_counters()), step_block_calls=1, step_sr_calls=1, step_host_fed_calls=1,
            grad_bf16_tensors=2, state_int8_tensors=2, ns_bf16_problems=4, weight_f32_tensors=2,
            host_pulled_bytes=2 * sum(r * c for r, c in shapes))
    q.qmuon_sync_status(sws)

    # ---- GRASP on two matrices ----
    gshapes = [(128, 192), (64, 64)]
    mats, keep = [], []
    for i, (r, c) in enumerate(gshapes):
        st = grasp.initial_state(r, c, np.random.default_rng(30 + i).standard_normal((c, 8)).astype(np.float32))
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
        d = [t(st.res), t(st.res_rmax), t(st.res_cmax), t(st.p), t(st.p_rmax), t(st.p_cmax), t(st.r),
             t(st.r_rmax), t(st.r_cmax), _grad(r, c, 40 + i)]
        keep.append(d)
        mats.append(q.grasp_matrix(r, c, *d))
    gws = torch.empty(q.qmuon_grasp_workspace_size(mats), dtype=torch.uint8, device="cuda")
    c0 = q.qmuon_get_counters()
    q.qmuon_grasp_step(mats, 0.9, gws)
    _expect(_delta(c0, q.qmuon_get_counters()), grasp_calls=1, grasp_matrices=2, grad_bf16_tensors=2)
    q.qmuon_sync_status(gws)

    # ---- a call that fails on the host adds nothing; reset zeroes every tally ----
    c0 = q.qmuon_get_counters()
    with pytest.raises(q.QmuonError):
        q.qmuon_step(splan, 0, 2, 0.95, 0.02, 0.01, weights, COEFFS, 5, sums, sws)   # t < 1
    _expect(_delta(c0, q.qmuon_get_counters()))
    q.qmuon_reset_counters()
    assert set(q.qmuon_get_counters().values()) == {0}
