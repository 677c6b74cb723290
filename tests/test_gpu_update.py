"""GPU parity of the momentum update and the MXFP8 carrier against the oracle.

Calls go through the C ABI (the ctypes binding).  Bars: q8 codes, absmax and
the stored momentum bit-exact; the carrier payload and scales bit-exact;
group sums and inverse norms within relative 1e-5 of the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import carrier, codec

from gpu_util import random_grad, to_oracle_grad, ulp_diff_bf16

pytestmark = pytest.mark.gpu

RAGGED = [(1, 17), (3, 100), (64, 256), (33, 1000), (256, 512), (1, 256), (2048, 300), (5, 7), (128, 4096)]


def _states(shapes, q8_kind, seed):
    out = []
    for i, (r, c) in enumerate(shapes):
        qs, a = workloads.random_state(workloads.Matrix("t", r, c), seed + i, q8_kind, device="cuda")
        # a few all-zero blocks (absmax 0 and zero codes)
        nb = a.numel()
        z = torch.arange(nb, device="cuda") % 7 == 3
        a[z] = 0.0
        zq = z.repeat_interleave(256)[: r * c]
        qs[zq] = 0 if q8_kind == "int8" else 128
        out.append((qs.contiguous(), a.contiguous()))
    return out


def _run(shapes, q8_kind, grad_dtype, beta, segments=None, n_groups=0, mode=0, seed=0):
    states = _states(shapes, q8_kind, 100 + seed)
    grads = [random_grad(r * c, grad_dtype, 1000 * seed + i) for i, (r, c) in enumerate(shapes)]
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, grad_dtype))
            for (s, a), g in zip(states, grads)]
    plan = q.qmuon_plan_create([(s, a, g, r, c) for (s, a), g, (r, c) in zip(states, grads, shapes)],
                               q8_kind, grad_dtype, segments=segments, n_groups=n_groups)
    G = q.qmuon_plan_info(plan)["n_groups"]
    sums = torch.full((G,), -1.0, device="cuda")
    inv = torch.full((G,), -1.0, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, beta, mode, sums, inv, ws)
    q.qmuon_sync_status(ws)
    segs = None if segments is None else [codec.NormSegment(*s) for s in segments]
    res, S, I, groups = codec.multi_update([h[0] for h in host], [h[1] for h in host], [h[2] for h in host], beta,
                                           grad_dtype=grad_dtype, q8_kind=q8_kind, segments=segs,
                                           n_groups=G)
    return states, grads, res, S, I, groups, sums, inv


def _check_state(states, grads, res, grad_dtype, exact_grad=True):
    for (s, a), g, r in zip(states, grads, res):
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
        got = to_oracle_grad(g, grad_dtype)
        if exact_grad:
            np.testing.assert_array_equal(got, r.grad)


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("grad_dtype", ["bf16", "f16", "f32"])
def test_update_ragged_multi_tensor(q8_kind, grad_dtype):
    states, grads, res, S, I, _, sums, inv = _run(RAGGED, q8_kind, grad_dtype, 0.95)
    _check_state(states, grads, res, grad_dtype)
    np.testing.assert_allclose(sums.cpu().numpy(), S, rtol=1e-5)
    np.testing.assert_allclose(inv.cpu().numpy(), I, rtol=1e-5)


@pytest.mark.parametrize("beta", [0.0, 0.5, 0.9, 1.0])
def test_update_betas(beta):
    states, grads, res, S, I, _, sums, inv = _run([(77, 300), (256, 256)], "int8", "bf16", beta, seed=3)
    _check_state(states, grads, res, "bf16")
    np.testing.assert_allclose(sums.cpu().numpy(), S, rtol=1e-5)


def test_update_interleaved_groups_many_waves():
    # fused-QKV-like interleaving (rows split 2:1:1 within every 4 rows), more
    # blocks than one wave of CTAs, several groups inside every CTA
    R, C = 2048, 2048
    shapes = [(R, C), (1024, 3000), (3, 256)]
    segs = [(0, r * C, C, [0, 0, 1, 2][r % 4]) for r in range(R)]
    segs.append((1, 0, 1024 * 3000, 3))
    segs.append((2, 256, 512, 4))      # tensor 2: block 0 ungrouped
    states, grads, res, S, I, _, sums, inv = _run(shapes, "int8", "bf16", 0.9, segments=segs, n_groups=5, seed=5)
    _check_state(states, grads, res, "bf16")
    np.testing.assert_allclose(sums.cpu().numpy(), S, rtol=1e-5)
    np.testing.assert_allclose(inv.cpu().numpy(), I, rtol=1e-5)


def test_update_inplace_normalize():
    shapes = [(64, 512), (10, 300)]
    segs = [(0, 0, 64 * 512, 0), (1, 0, 3000, 1)]
    states, grads, res, S, I, groups, sums, inv = _run(shapes, "int8", "bf16", 0.9, segments=segs, n_groups=2,
                                                       mode=1, seed=9)
    for (s, a), g, r, gid in zip(states, grads, res, groups):
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8)
        # the scale is the GPU's own inverse norm (within 1e-5 of the oracle's);
        # with it the stored value is exact, with the oracle's it is within 1 ulp
        expect = codec.normalize_inplace(r.grad, gid, inv.cpu().numpy())
        np.testing.assert_array_equal(to_oracle_grad(g, "bf16"), expect)
        expect2 = codec.normalize_inplace(r.grad, gid, I)
        assert ulp_diff_bf16(to_oracle_grad(g, "bf16"), expect2) <= 1


def test_update_three_step_recurrence_c1():
    # the 512x512 workload: zero state, N(0,1e-3^2) grads, three steps
    w = workloads.get(1)
    m = w.matrices[0]
    qs, a = workloads.zero_state(m, "int8", device="cuda")
    hq, ha = qs.cpu().numpy(), a.cpu().numpy()
    for step in range(1, 4):
        g = workloads.make_grad(w, 0, step, device="cuda")
        hg = to_oracle_grad(g, "bf16")
        plan = q.qmuon_plan_create([(qs, a, g, m.rows, m.cols)])
        ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
        sums = torch.zeros(1, device="cuda")
        q.qmuon_update_multi_normalize_groups(plan, w.beta, 2, sums, torch.zeros(1, device="cuda"), ws)
        r = codec.momentum_update(hq, ha, hg, w.beta)
        np.testing.assert_array_equal(qs.cpu().numpy(), r.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
        np.testing.assert_array_equal(to_oracle_grad(g, "bf16"), r.grad)
        np.testing.assert_allclose(sums.item(), r.block_sumsq.sum(), rtol=1e-5)
        hq, ha = r.q8, r.absmax


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_long_chain_bit_exact_and_drift_bounded(q8_kind):
    # 40 updates of one plan in a row, each bit-exact against the oracle's
    # step from the oracle's own previous state (so no error can build up on
    # either side), and the dequantised state within max(absmax)/254/(1-beta)
    # of the exact fp64 EMA of the same gradients at every step
    shapes = [(33, 1000), (1, 17), (64, 256)]
    beta, steps = 0.95, 40
    states = [workloads.zero_state(workloads.Matrix("t", r, c), q8_kind, device="cuda") for r, c in shapes]
    grads = [torch.empty(r * c, dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    plan = q.qmuon_plan_create([(s, a, g, r, c) for (s, a), g, (r, c) in zip(states, grads, shapes)],
                               q8_kind, "bf16")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    sums = torch.zeros(len(shapes), device="cuda")
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy()) for s, a in states]
    exact = [np.zeros(r * c) for r, c in shapes]
    amax_seen = [np.zeros((r * c + 255) // 256) for r, c in shapes]
    bias = [random_grad(r * c, "f32", 77 + i) for i, (r, c) in enumerate(shapes)]
    for t in range(steps):
        for i, g in enumerate(grads):
            g.copy_((bias[i] + random_grad(g.numel(), "f32", 1000 + 10 * t + i)).to(torch.bfloat16))
        hg = [to_oracle_grad(g, "bf16") for g in grads]
        q.qmuon_update_multi_normalize_groups(plan, beta, 0, sums, None, ws)
        q.qmuon_sync_status(ws)
        res, S, _, _ = codec.multi_update([h[0] for h in host], [h[1] for h in host], hg, beta, q8_kind=q8_kind)
        np.testing.assert_allclose(sums.cpu().numpy(), S, rtol=1e-5, err_msg=str(t))
        for i, ((s, a), r) in enumerate(zip(states, res)):
            np.testing.assert_array_equal(s.cpu().numpy(), r.q8, err_msg=f"step {t} tensor {i}")
            np.testing.assert_array_equal(a.cpu().numpy(), r.absmax, err_msg=f"step {t} tensor {i}")
            np.testing.assert_array_equal(to_oracle_grad(grads[i], "bf16"), r.grad, err_msg=f"step {t} tensor {i}")
            exact[i] = beta * exact[i] + (1.0 - beta) * codec.f32_from_bf16_bits(hg[i]).astype(np.float64)
            amax_seen[i] = np.maximum(amax_seen[i], r.absmax)
            drift = codec.dequantize(r.q8, r.absmax, q8_kind).astype(np.float64) - exact[i]
            bound = np.repeat(amax_seen[i] / 254.0 / (1.0 - beta), 256)[:drift.size] * (1.0 + 1e-5) \
                + 1e-6 * np.abs(exact[i])
            assert np.all(np.abs(drift) <= bound), (t, i)
        host = [(r.q8, r.absmax) for r in res]


def test_update_full_size_decoder_sampled():
    # the 24-matrix 2048-hidden workload at full size: every block checked on a
    # sample, group sums of three whole tensors against the oracle
    w = workloads.get(2)
    states, grads, host = [], [], []
    rng = np.random.default_rng(0)
    for i, m in enumerate(w.matrices):
        qs, a = workloads.random_state(m, 500 + i, device="cuda")
        g = workloads.make_grad(w, i, 1, device="cuda")
        states.append((qs, a))
        grads.append(g)
    # sampled blocks: copy their inputs before the update
    picks = []
    for i, m in enumerate(w.matrices):
        nb = (m.numel + 255) // 256
        for b in rng.choice(nb, size=40, replace=False):
            sl = slice(int(b) * 256, int(b) * 256 + 256)
            picks.append((i, int(b), states[i][0][sl].cpu().numpy().copy(), states[i][1][int(b):int(b) + 1].cpu().numpy().copy(),
                          to_oracle_grad(grads[i].reshape(-1)[sl], "bf16")))
    whole = [0, 4, 6]
    whole_in = {i: (states[i][0].cpu().numpy().copy(), states[i][1].cpu().numpy().copy(),
                    to_oracle_grad(grads[i], "bf16")) for i in whole}
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, w.matrices)])
    sums = torch.zeros(len(w.matrices), device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, w.beta, 0, sums, None, ws)
    q.qmuon_sync_status(ws)
    for i, b, hq, ha, hg in picks:
        r = codec.momentum_update(hq, ha, hg, w.beta)
        sl = slice(b * 256, b * 256 + 256)
        np.testing.assert_array_equal(states[i][0][sl].cpu().numpy(), r.q8)
        assert states[i][1][b].item() == r.absmax[0]
        np.testing.assert_array_equal(to_oracle_grad(grads[i].reshape(-1)[sl], "bf16"), r.grad)
    for i in whole:
        r = codec.momentum_update(*whole_in[i], w.beta)
        np.testing.assert_allclose(sums[i].item(), r.block_sumsq.sum(), rtol=1e-5)


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("shape", [(64, 4096), (37, 96), (1, 32), (300, 1024)])
def test_carrier_parity(q8_kind, shape):
    rows, cols = shape
    m = workloads.Matrix("t", rows, cols)
    qs, a = workloads.random_state(m, 11, q8_kind, device="cuda")
    g = random_grad(rows * cols, "bf16", 12)
    g_before = g.clone()
    hq, ha, hg = qs.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, "bf16")
    payload = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows * (cols // 32), dtype=torch.uint8, device="cuda")
    inv = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_carrier_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier(qs, a, g, rows, cols, q8_kind, "bf16", 0.95, payload, scale, inv, ws)
    q.qmuon_sync_status(ws)
    r = carrier.carrier_update(hq, ha, hg, 0.95, rows, cols, q8_kind=q8_kind)
    np.testing.assert_array_equal(qs.cpu().numpy(), r.q8)
    np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
    np.testing.assert_array_equal(scale.cpu().numpy().reshape(rows, cols // 32), r.scale_inv)
    np.testing.assert_array_equal(payload.cpu().numpy().reshape(rows, cols), r.payload)
    np.testing.assert_allclose(inv.item(), r.inv_norm, rtol=1e-5)
    assert torch.equal(g, g_before)   # the gradient is read only


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_carrier_multi_matches_oracle(q8_kind, grad_dtype):
    # one launch over tensors of several shapes (ragged rows, blocks that span
    # tensors): every tensor as the oracle's single-tensor carrier
    shapes = [(64, 4096), (37, 96), (1, 32), (300, 1024), (5, 224)]
    states = [workloads.random_state(workloads.Matrix("t", r, c), 90 + i, q8_kind, device="cuda")
              for i, (r, c) in enumerate(shapes)]
    grads = [random_grad(r * c, grad_dtype, 20 + i) for i, (r, c) in enumerate(shapes)]
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, grad_dtype))
            for (s, a), g in zip(states, grads)]
    before = [g.clone() for g in grads]
    plan = q.qmuon_plan_create([(s, a, g, r, c) for (s, a), g, (r, c) in zip(states, grads, shapes)],
                               q8_kind, grad_dtype)
    payloads = [torch.empty(r * c, dtype=torch.uint8, device="cuda") for r, c in shapes]
    scales = [torch.empty(r * (c // 32), dtype=torch.uint8, device="cuda") for r, c in shapes]
    inv = torch.zeros(len(shapes), device="cuda")
    sums = torch.zeros(len(shapes), device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier_multi(plan, 0.95, payloads, scales, inv, ws, group_sumsq=sums)
    q.qmuon_sync_status(ws)
    for i, ((r, c), (s, a), h) in enumerate(zip(shapes, states, host)):
        ref = carrier.carrier_update(h[0], h[1], h[2], 0.95, r, c, q8_kind=q8_kind, grad_dtype=grad_dtype)
        np.testing.assert_array_equal(s.cpu().numpy(), ref.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), ref.absmax)
        np.testing.assert_array_equal(scales[i].cpu().numpy().reshape(r, c // 32), ref.scale_inv)
        np.testing.assert_array_equal(payloads[i].cpu().numpy().reshape(r, c), ref.payload)
        np.testing.assert_allclose(inv[i].item(), ref.inv_norm, rtol=1e-5)
        assert torch.equal(grads[i], before[i])   # gradients are read only


def test_carrier_multi_rejects_unaligned_columns():
    m = workloads.Matrix("t", 4, 40)
    s, a = workloads.random_state(m, 1, device="cuda")
    g = random_grad(m.numel, "bf16", 2)
    plan = q.qmuon_plan_create([(s, a, g, 4, 40)])
    pay = torch.empty(160, dtype=torch.uint8, device="cuda")
    sc = torch.empty(8, dtype=torch.uint8, device="cuda")
    inv = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_update_mxfp8_carrier_multi(plan, 0.9, [pay], [sc], inv, ws)
    assert e.value.status == q.QMUON_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["update", "carrier"])
def test_update_and_carrier_do_not_depend_on_workspace_contents(entry):
    # the same multi-tensor launch with the workspace zeroed and with every
    # byte 0xFF (NaN partial sums, garbage tables) leaves bit-identical codes,
    # absmax, momenta or carriers and group sums: each workspace value is
    # written before it is read
    shapes = [(64, 4096), (37, 96), (300, 1024), (5, 224), (2048, 300)]
    if entry == "carrier":
        shapes = [(r, c) for r, c in shapes if c % 32 == 0]
    outs = []
    for fill in (0x00, 0xFF):
        states = _states(shapes, "int8", 300)
        grads = [random_grad(r * c, "bf16", 310 + i) for i, (r, c) in enumerate(shapes)]
        plan = q.qmuon_plan_create([(s, a, g, r, c) for (s, a), g, (r, c) in zip(states, grads, shapes)],
                                   "int8", "bf16")
        ws = torch.full((q.qmuon_workspace_size(plan),), fill, dtype=torch.uint8, device="cuda")
        G = max(q.qmuon_plan_info(plan)["n_groups"], len(shapes))
        sums = torch.zeros(G, device="cuda")
        inv = torch.zeros(G, device="cuda")
        extra = []
        if entry == "update":
            q.qmuon_update_multi_normalize_groups(plan, 0.9, 0, sums, inv, ws)
        else:
            pays = [torch.empty(r * c, dtype=torch.uint8, device="cuda") for r, c in shapes]
            scs = [torch.empty(r * (c // 32), dtype=torch.uint8, device="cuda") for r, c in shapes]
            q.qmuon_update_mxfp8_carrier_multi(plan, 0.9, pays, scs, inv, ws, group_sumsq=sums)
            extra = pays + scs
        q.qmuon_sync_status(ws)
        outs.append([x for s in states for x in s] + grads + extra + [sums, inv])
    for a, b in zip(*outs):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
