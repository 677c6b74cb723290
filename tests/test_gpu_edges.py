"""Edge cases of the update and the step: empty tensors inside a plan (their
groups sum to 0, so the inverse norm is 1 / (0 + 1e-7)), a plan of only
empty tensors (rejected: a plan holds at least one block), and a tensor of more than 2^31 elements, whose blocks around
element 2^31 and at its end are checked bit-exact against the oracle (64-bit
element and block indexing).  Failure reporting: a status recorded in a
workspace header (injected from the host) comes back from qmuon_sync_status
with its site, and is cleared by the read."""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import codec, muonbp

from gpu_util import random_grad, to_oracle_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)


def _tensors(shapes, seed):
    out = []
    for i, (r, c) in enumerate(shapes):
        m = workloads.Matrix(f"m{i}", r, c)
        if m.numel:
            qs, a = workloads.random_state(m, seed + i, device="cuda")
            g = random_grad(m.numel, "bf16", seed + 50 + i).reshape(r, c)
        else:   # empty: valid (aligned) pointers that are never touched
            qs = torch.zeros(16, dtype=torch.int8, device="cuda")
            a = torch.zeros(4, device="cuda")
            g = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
        out.append((m, qs, a, g))
    return out


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_empty_tensors_in_a_plan(mode):
    shapes = [(0, 128), (37, 96), (64, 0), (256, 256)]
    ts = _tensors(shapes, 10)
    host = [(qs.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, "bf16")) for m, qs, a, g in ts
            if m.numel]
    plan = q.qmuon_plan_create([(qs, a, g, m.rows, m.cols) for m, qs, a, g in ts], "int8", "bf16")
    sums = torch.full((len(shapes),), -1.0, device="cuda")
    inv = torch.full((len(shapes),), -1.0, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, 0.9, mode, sums, inv, ws)
    q.qmuon_sync_status(ws)
    res = [codec.momentum_update(hq, ha, hg, 0.9) for hq, ha, hg in host]
    live = [t for t in ts if t[0].numel]
    for (m, qs, a, g), r in zip(live, res):
        np.testing.assert_array_equal(qs.cpu().numpy(), r.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
    S = sums.cpu().numpy()
    assert S[0] == 0.0 and S[2] == 0.0
    np.testing.assert_allclose(S[[1, 3]], [r.block_sumsq.sum() for r in res], rtol=1e-5)
    np.testing.assert_allclose(inv.cpu().numpy()[[0, 2]], [1e7, 1e7], rtol=1e-6)


def test_plan_of_only_empty_tensors_is_rejected():
    # a plan needs at least one quantization block
    ts = _tensors([(0, 64), (16, 0)], 20)
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_plan_create([(qs, a, g, m.rows, m.cols) for m, qs, a, g in ts], "int8", "bf16")
    assert e.value.status == q.QMUON_ERR_INVALID_ARGUMENT


def test_step_with_an_empty_tensor():
    shapes = [(256, 512), (0, 512), (128, 512)]
    ts = _tensors(shapes, 30)
    weights = [(torch.randn(m.rows, m.cols, device="cuda") * 0.02) if m.numel else None for m, *_ in ts]
    host = [muonbp.MatrixState(m.rows, m.cols, qs.cpu().numpy(), a.cpu().numpy(), w.cpu().numpy())
            for (m, qs, a, g), w in zip(ts, weights) if m.numel]
    grads_h = [to_oracle_grad(g, "bf16") for m, qs, a, g in ts if m.numel]
    plan = q.qmuon_plan_create([(qs, a, g, m.rows, m.cols) for m, qs, a, g in ts], "int8", "bf16", tile=(1, 2))
    info = q.qmuon_plan_info(plan)
    sums = torch.zeros(max(info["n_full_groups"], info["n_block_groups"]), device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    q.qmuon_step(plan, 1, 2, 0.95, 0.02, 0.01, [w if w is not None else 0 for w in weights], COEFFS, 5, sums, ws)
    q.qmuon_sync_status(ws)
    new, U, inf = muonbp.muonbp_step(1, 2, host, grads_h, 0.95, 0.02, 0.01, tile=(1, 2))
    for (m, qs, a, g), st in zip([t for t in ts if t[0].numel], new):
        np.testing.assert_array_equal(qs.cpu().numpy(), st.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), st.absmax)


def test_tensor_past_2_pow_31_elements():
    rows, cols = 32769, 65536                       # 2,147,549,184 elements
    n = rows * cols
    assert n > 2 ** 31
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    qs = torch.randint(-127, 128, (n,), generator=gen, device="cuda", dtype=torch.int8)
    nb = (n + 255) // 256
    a = torch.exp(torch.empty(nb, device="cuda").uniform_(-9.0, 3.0, generator=gen))
    g = torch.randn(n, generator=gen, device="cuda", dtype=torch.bfloat16)
    picks = [0, 2 ** 31 // 256 - 1, 2 ** 31 // 256, 2 ** 31 // 256 + 1, nb // 2, nb - 1]
    ins = {b: (qs[b * 256:(b + 1) * 256].cpu().numpy().copy(), a[b:b + 1].cpu().numpy().copy(),
               to_oracle_grad(g[b * 256:(b + 1) * 256], "bf16")) for b in picks}
    plan = q.qmuon_plan_create([(qs, a, g, rows, cols)], "int8", "bf16")
    sums = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, 0.9, 0, sums, None, ws)
    q.qmuon_sync_status(ws)
    for b in picks:
        r = codec.momentum_update(*ins[b], 0.9)
        np.testing.assert_array_equal(qs[b * 256:(b + 1) * 256].cpu().numpy(), r.q8, err_msg=str(b))
        assert a[b].item() == r.absmax[0]
        np.testing.assert_array_equal(to_oracle_grad(g[b * 256:(b + 1) * 256], "bf16"), r.grad, err_msg=str(b))
    assert np.isfinite(sums.item()) and sums.item() > 0


@pytest.mark.parametrize("status,site", [(q.QMUON_ERR_TIMEOUT, 0x1300), (q.QMUON_ERR_INVALID_ARGUMENT, 0x2003)])
def test_sync_status_reports_and_clears_a_recorded_failure(status, site):
    # a kernel records a failure as (status, site) in the workspace header's
    # first two words; injected from the host here, with no kernel made to fail
    ts = _tensors([(64, 256)], 40)
    plan = q.qmuon_plan_create([(qs, a, g, m.rows, m.cols) for m, qs, a, g in ts], "int8", "bf16")
    ws = torch.zeros(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_sync_status(ws)   # a clean header
    ws[:8].view(torch.int32).copy_(torch.tensor([status, site], dtype=torch.int32))
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_sync_status(ws)
    assert e.value.status == status
    assert f"0x{site:x}" in q.qmuon_last_error()
    assert ws[:8].view(torch.int32).cpu().tolist() == [0, 0]   # cleared by the read
    q.qmuon_sync_status(ws)
    # the next call on the workspace starts from a clean header and succeeds
    inv = torch.zeros(1, device="cuda")
    ws[:8].view(torch.int32).copy_(torch.tensor([status, site], dtype=torch.int32))
    q.qmuon_update_multi_normalize_groups(plan, 0.9, 2, None, inv, ws)
    q.qmuon_sync_status(ws)
