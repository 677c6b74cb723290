"""GPU parity of the stochastic requantisation against the oracle.

q8 codes, absmax and the stored momentum bit-exact (the generator and the
floor are exact on both sides), for every storage and gradient type, ragged
tensors, seeds and steps above 2^32, and through qmuon_step with the plan's
stochastic rounding switched on.
"""

import math

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import codec

from gpu_util import random_grad, to_oracle_grad

pytestmark = pytest.mark.gpu

RAGGED = [(1, 17), (3, 100), (64, 256), (33, 1000), (256, 512), (5, 7), (128, 4096)]


def _states(shapes, q8_kind, seed):
    return [workloads.random_state(workloads.Matrix("t", r, c), seed + i, q8_kind, device="cuda")
            for i, (r, c) in enumerate(shapes)]


def _run_sr(shapes, q8_kind, grad_dtype, beta, seed, step, mode=2):
    states = _states(shapes, q8_kind, 300)
    grads = [random_grad(r * c, grad_dtype, 40 + i) for i, (r, c) in enumerate(shapes)]
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, grad_dtype))
            for (s, a), g in zip(states, grads)]
    plan = q.qmuon_plan_create([(s, a, g, r, c) for (s, a), g, (r, c) in zip(states, grads, shapes)],
                               q8_kind, grad_dtype)
    G = q.qmuon_plan_info(plan)["n_groups"]
    sums = torch.zeros(G, device="cuda")
    inv = torch.zeros(G, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups_sr(plan, beta, mode, seed, step, sums, inv, ws)
    q.qmuon_sync_status(ws)
    res, S, I, _ = codec.multi_update([h[0] for h in host], [h[1] for h in host], [h[2] for h in host], beta,
                                      grad_dtype=grad_dtype, q8_kind=q8_kind, n_groups=G,
                                      sr_seed=seed, sr_step=step)
    for (s, a), g, r in zip(states, grads, res):
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
        np.testing.assert_array_equal(to_oracle_grad(g, grad_dtype), r.grad)
    np.testing.assert_allclose(sums.cpu().numpy(), S, rtol=1e-5)
    np.testing.assert_allclose(inv.cpu().numpy(), I, rtol=1e-5)


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("grad_dtype", ["bf16", "f16", "f32"])
def test_sr_ragged_multi_tensor(q8_kind, grad_dtype):
    _run_sr(RAGGED, q8_kind, grad_dtype, 0.95, seed=20260101, step=7)


@pytest.mark.parametrize("seed,step", [(0, 1), ((1 << 40) + 12345, (1 << 33) + 5), (0xFFFFFFFFFFFFFFFF, 1 << 32)])
def test_sr_seed_and_step_words(seed, step):
    _run_sr([(77, 300), (256, 256)], "int8", "bf16", 0.9, seed=seed, step=step)


def test_sr_large_tensor():
    # 16.8M elements: counters far from zero, several waves of CTAs
    _run_sr([(4096, 4096), (1, 300)], "int8", "bf16", 0.95, seed=3, step=2, mode=0)


def test_sr_step_entry():
    # qmuon_step with the plan's stochastic rounding: the update of step t
    # draws with step word t and the tensor's index
    shapes = [(512, 2048), (256, 2048)]
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    states = [workloads.random_state(m, 60 + i, device="cuda") for i, m in enumerate(mats)]
    weights = [(torch.randn(m.rows, m.cols, device="cuda") * 0.02).contiguous() for m in mats]
    grads = [random_grad(m.numel, "bf16", 70 + i).reshape(m.rows, m.cols) for i, m in enumerate(mats)]
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, "bf16"))
            for (s, a), g in zip(states, grads)]
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, mats)],
                               "int8", "bf16", tile=(1, 8))
    q.qmuon_plan_set_stochastic_rounding(plan, True, seed=99)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    t = 3
    sums = torch.zeros(q.qmuon_plan_info(plan)["n_block_groups"], device="cuda")
    q.qmuon_step(plan, t, 5, 0.95, 0.02, 0.02 / math.sqrt(8), weights, workloads.COEFFS, 5, sums, ws)
    q.qmuon_sync_status(ws)
    for i, ((s, a), h) in enumerate(zip(states, host)):
        r = codec.momentum_update(h[0], h[1], h[2], 0.95, rounding=codec.StochasticRounding(99, t, i))
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8)
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax)
    # switched off again: nearest rounding
    q.qmuon_plan_set_stochastic_rounding(plan, False)
    host2 = [(s.cpu().numpy().copy(), a.cpu().numpy().copy()) for s, a in states]
    for g, i in zip(grads, range(2)):
        g.copy_(random_grad(g.numel(), "bf16", 80 + i).reshape(g.shape))
    gh = [to_oracle_grad(g, "bf16") for g in grads]
    q.qmuon_step(plan, t + 1, 5, 0.95, 0.02, 0.02 / math.sqrt(8), weights, workloads.COEFFS, 5, sums, ws)
    q.qmuon_sync_status(ws)
    for (s, a), h, g in zip(states, host2, gh):
        r = codec.momentum_update(h[0], h[1], g, 0.95)
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8)


def test_sr_rejects_bad_switch():
    m = workloads.Matrix("t", 16, 256)
    s, a = workloads.random_state(m, 1, device="cuda")
    g = random_grad(m.numel, "bf16", 2)
    plan = q.qmuon_plan_create([(s, a, g, 16, 256)])
    assert q.lib().qmuon_plan_set_stochastic_rounding(plan.handle, 2, 0) == q.QMUON_ERR_INVALID_ARGUMENT
    assert q.lib().qmuon_plan_set_stochastic_rounding(None, 1, 0) == q.QMUON_ERR_INVALID_ARGUMENT
