"""GPU parity of ``qmuon_step_from_host``: the MuonBP step fed from host
gradients, copied in on a second stream while the previous step computes.

Two plans share one q8 state, one set of weights and one workspace, and have
separate gradient buffers; steps alternate between them and are enqueued
without any synchronisation in between.  The oracle runs the same steps in
order.  The momentum never depends on the weights or on U, so codes, absmax
and every step's group sums (read back to host memory) must match after the
last step: codes and absmax bit-exactly, sums within 1e-5.  The U left in each
plan's buffers is that of its last step (2e-2 / 0.999), and the weights moved
by the sum of the applied updates.
"""

import math

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import codec, muonbp

from gpu_util import bf16_to_f64, min_row_cos, random_grad, rel_fro, to_oracle_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)


def _setup(shapes, tile, seed):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    states = [workloads.random_state(m, seed + i, device="cuda") for i, m in enumerate(mats)]
    weights = [(torch.randn(m.rows, m.cols, device="cuda") * 0.02).contiguous() for m in mats]
    bufs = [[torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device="cuda") for m in mats] for _ in range(2)]
    plans = [q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, b, mats)],
                                 "int8", "bf16", tile=tile) for b in bufs]
    host = [muonbp.MatrixState(m.rows, m.cols, s[0].cpu().numpy().copy(), s[1].cpu().numpy().copy(),
                               w.cpu().numpy().copy()) for m, s, w in zip(mats, states, weights)]
    return mats, states, weights, bufs, plans, host


@pytest.mark.parametrize("shapes,tile,P,steps", [
    ([(512, 2048), (256, 1024), (1024, 512)], (1, 2), 2, 4),
    ([(300, 520), (520, 136), (8, 16)], (1, 1), 1, 3),
])
def test_overlapped_host_steps_match_oracle(shapes, tile, P, steps):
    mats, states, weights, bufs, plans, host = _setup(shapes, tile, 60)
    ws = torch.empty(q.qmuon_workspace_size(plans[0], q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    for p in plans:
        q.qmuon_step_prepare(p, weights, ws)
    info = q.qmuon_plan_info(plans[0])
    eta_full, eta_block = 0.02, 0.02 / math.sqrt(tile[0] * tile[1])
    # every step's gradients in page-locked host memory, kept alive until the end
    grads_h = [[random_grad(m.numel, "bf16", 300 + 10 * t + i).reshape(m.rows, m.cols).cpu().pin_memory()
                for i, m in enumerate(mats)] for t in range(1, steps + 1)]
    sums_h = [torch.zeros(max(info["n_full_groups"], info["n_block_groups"])).pin_memory() for _ in range(steps)]
    sums_d = torch.zeros(max(info["n_full_groups"], info["n_block_groups"]), device="cuda")
    w0 = [w.cpu().numpy().astype(np.float64) for w in weights]
    copy_stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    for t in range(1, steps + 1):
        q.qmuon_step_from_host(plans[(t - 1) % 2], t, P, 0.95, eta_full, eta_block, weights, COEFFS, 5,
                               grads_h[t - 1], sums_h[t - 1], sums_d, ws, copy_stream=copy_stream)
    q.qmuon_sync_status(ws)
    torch.cuda.synchronize()

    U_last = {}
    for t in range(1, steps + 1):
        gh = [to_oracle_grad(g, "bf16") for g in grads_h[t - 1]]
        host, U, inf = muonbp.muonbp_step(t, P, host, gh, 0.95, eta_full, eta_block, tile=tile)
        np.testing.assert_allclose(sums_h[t - 1][:inf["n_groups"]].numpy(), inf["S"], rtol=1e-5, err_msg=str(t))
        U_last[(t - 1) % 2] = (t, U, inf["full"])
    for i, m in enumerate(mats):
        np.testing.assert_array_equal(states[i][0].cpu().numpy(), host[i].q8)
        np.testing.assert_array_equal(states[i][1].cpu().numpy(), host[i].absmax)
        dW = weights[i].cpu().numpy().astype(np.float64) - w0[i]
        dW_ref = host[i].weight.astype(np.float64) - w0[i]
        assert rel_fro(dW, dW_ref) <= 2e-2, m
    for b, (t, U, full) in U_last.items():
        for i, m in enumerate(mats):
            got = bf16_to_f64(bufs[b][i])
            ref = codec.f32_from_bf16_bits(U[i]).astype(np.float64)
            th, tw = (m.rows, m.cols) if full else (m.rows // tile[0], m.cols // tile[1])
            for bi in range(m.rows // th):
                for bj in range(m.cols // tw):
                    sl = (slice(bi * th, (bi + 1) * th), slice(bj * tw, (bj + 1) * tw))
                    assert rel_fro(got[sl], ref[sl]) <= 2e-2 and min_row_cos(got[sl], ref[sl]) >= 0.999, (t, m)


def test_same_stream_and_pageable_host_memory():
    # no copy stream and pageable host gradients: the copies run in order on
    # the step's stream; the result equals the oracle's step exactly where the
    # arithmetic is exact
    mats, states, weights, bufs, plans, host = _setup([(256, 512), (128, 256)], (1, 1), 80)
    ws = torch.empty(q.qmuon_workspace_size(plans[0], q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    gh_t = [random_grad(m.numel, "bf16", 500 + i).reshape(m.rows, m.cols).cpu() for i, m in enumerate(mats)]
    sums_h = torch.full((2,), -1.0)
    w_before = [w.cpu().numpy() for w in weights]
    q.qmuon_step_from_host(plans[0], 1, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, gh_t, sums_h, None, ws)
    q.qmuon_sync_status(ws)
    host, U, inf = muonbp.muonbp_step(1, 1, host, [to_oracle_grad(g, "bf16") for g in gh_t], 0.9, 0.02, 0.02,
                                      tile=(1, 1))
    np.testing.assert_allclose(sums_h.numpy(), inf["S"], rtol=1e-5)
    for i, m in enumerate(mats):
        np.testing.assert_array_equal(states[i][0].cpu().numpy(), host[i].q8)
        np.testing.assert_array_equal(states[i][1].cpu().numpy(), host[i].absmax)
        u32 = bufs[0][i].float().cpu().numpy()
        expect = (w_before[i] - (np.float32(0.02) * u32).astype(np.float32)).astype(np.float32)
        np.testing.assert_array_equal(weights[i].cpu().numpy(), expect)


def test_rejects_missing_host_gradient():
    mats, states, weights, bufs, plans, host = _setup([(64, 64), (64, 128)], (1, 1), 90)
    ws = torch.empty(q.qmuon_workspace_size(plans[0], q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    g0 = torch.zeros(64, 64, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_step_from_host(plans[0], 1, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, [g0, 0], None, None, ws)
    assert e.value.status == q.QMUON_ERR_INVALID_ARGUMENT


def test_page_locked_pull_and_copy_paths_in_one_step():
    # page-locked 16-byte aligned gradients are read by the device's own loads
    # (host_pulled_bytes), pageable ones and a page-locked view that starts 2
    # bytes into its buffer are copied (host_copied_bytes); the step equals the
    # oracle's where its arithmetic is exact, as with every gradient copied
    shapes = [(256, 512), (128, 256), (64, 192)]
    mats, states, weights, bufs, plans, host = _setup(shapes, (1, 1), 95)
    ws = torch.empty(q.qmuon_workspace_size(plans[0], q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    g = [random_grad(m.numel, "bf16", 700 + i).reshape(m.rows, m.cols).cpu() for i, m in enumerate(mats)]
    pinned = g[0].pin_memory()
    pageable = g[1].clone()
    wide = torch.empty(mats[2].numel + 8, dtype=torch.bfloat16).pin_memory()
    wide[1:1 + mats[2].numel] = g[2].reshape(-1)
    shifted = wide[1:1 + mats[2].numel].view(mats[2].rows, mats[2].cols)
    assert shifted.data_ptr() % 16 == 2
    sums_h = torch.full((3,), -1.0)
    w_before = [w.cpu().numpy() for w in weights]
    before = q.qmuon_get_counters()
    q.qmuon_step_from_host(plans[0], 1, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, [pinned, pageable, shifted], sums_h,
                           None, ws)
    q.qmuon_sync_status(ws)
    after = q.qmuon_get_counters()
    assert after["host_pulled_bytes"] - before["host_pulled_bytes"] == 2 * mats[0].numel
    assert after["host_copied_bytes"] - before["host_copied_bytes"] == 2 * (mats[1].numel + mats[2].numel)
    host, U, inf = muonbp.muonbp_step(1, 1, host, [to_oracle_grad(x, "bf16") for x in g], 0.9, 0.02, 0.02,
                                      tile=(1, 1))
    np.testing.assert_allclose(sums_h.numpy(), inf["S"], rtol=1e-5)
    for i, m in enumerate(mats):
        np.testing.assert_array_equal(states[i][0].cpu().numpy(), host[i].q8)
        np.testing.assert_array_equal(states[i][1].cpu().numpy(), host[i].absmax)
        u32 = bufs[0][i].float().cpu().numpy()
        expect = (w_before[i] - (np.float32(0.02) * u32).astype(np.float32)).astype(np.float32)
        np.testing.assert_array_equal(weights[i].cpu().numpy(), expect)

    # the plan told to copy: the same page-locked buffers go through the copy engines
    q.qmuon_plan_set_host_ingest(plans[0], q.QMUON_INGEST_COPY)
    g2 = [random_grad(m.numel, "bf16", 710 + i).reshape(m.rows, m.cols).cpu().pin_memory() for i, m in enumerate(mats)]
    before = q.qmuon_get_counters()
    q.qmuon_step_from_host(plans[0], 2, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, g2, sums_h, None, ws)
    q.qmuon_sync_status(ws)
    after = q.qmuon_get_counters()
    assert after["host_pulled_bytes"] == before["host_pulled_bytes"]
    assert after["host_copied_bytes"] - before["host_copied_bytes"] == 2 * sum(m.numel for m in mats)
    host, U, inf = muonbp.muonbp_step(2, 1, host, [to_oracle_grad(x, "bf16") for x in g2], 0.9, 0.02, 0.02,
                                      tile=(1, 1))
    np.testing.assert_allclose(sums_h.numpy(), inf["S"], rtol=1e-5)
    for i, m in enumerate(mats):
        np.testing.assert_array_equal(states[i][0].cpu().numpy(), host[i].q8)
        np.testing.assert_array_equal(states[i][1].cpu().numpy(), host[i].absmax)
