"""Checkpoint and resume.  The optimizer state is the caller's q8 codes,
absmax and fp32 master weights; a plan and a workspace carry nothing one step
needs from an earlier one.  A run saved after step 3 and restored into fresh
buffers, a fresh plan and a fresh workspace continues bit-identically through
the next full and block steps, with nearest and with stochastic
requantisation (whose Philox counter is (element, tensor, step) under the
plan's seed)."""

import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads

from gpu_util import random_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)
SHAPES = [(512, 512), (256, 1024), (300, 520), (130, 136)]
P = 3


def _grads(t):
    return [random_grad(r * c, "bf16", 1000 + 10 * t + i).reshape(r, c) for i, (r, c) in enumerate(SHAPES)]


def _make(states, weights, sr):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(SHAPES)]
    grads = [torch.empty(r, c, dtype=torch.bfloat16, device="cuda") for r, c in SHAPES]
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, mats)], "int8", "bf16")
    if sr:
        q.qmuon_plan_set_stochastic_rounding(plan, True, 0x1234_5678_9ABC)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    info = q.qmuon_plan_info(plan)
    sums = torch.zeros(max(info["n_full_groups"], info["n_block_groups"]), device="cuda")
    return plan, grads, ws, sums


def _run(plan, grads, ws, sums, weights, ts):
    for t in ts:
        for g, src in zip(grads, _grads(t)):
            g.copy_(src)
        q.qmuon_step(plan, t, P, 0.95, 0.02, 0.01, weights, COEFFS, 5, sums, ws)
        q.qmuon_sync_status(ws)


@pytest.mark.parametrize("sr", [False, True])
def test_resume_continues_bit_identically(sr):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(SHAPES)]
    states = [workloads.random_state(m, 5 + i, device="cuda") for i, m in enumerate(mats)]
    weights = [(torch.randn(r, c, device="cuda") * 0.02).contiguous() for r, c in SHAPES]
    plan, grads, ws, sums = _make(states, weights, sr)
    _run(plan, grads, ws, sums, weights, range(1, 4))
    saved = ([(s.cpu().clone(), a.cpu().clone()) for s, a in states], [w.cpu().clone() for w in weights])
    _run(plan, grads, ws, sums, weights, range(4, 7))

    # restore into fresh device buffers, a fresh plan and a fresh workspace
    states2 = [(s.cuda(), a.cuda()) for s, a in saved[0]]
    weights2 = [w.cuda() for w in saved[1]]
    plan2, grads2, ws2, sums2 = _make(states2, weights2, sr)
    _run(plan2, grads2, ws2, sums2, weights2, range(4, 7))

    for (s, a), (s2, a2) in zip(states, states2):
        assert torch.equal(s, s2) and torch.equal(a, a2)
    for w, w2 in zip(weights, weights2):
        assert torch.equal(w, w2)
    for g, g2 in zip(grads, grads2):   # the last step's U
        assert torch.equal(g.view(torch.int16), g2.view(torch.int16))
    assert torch.equal(sums, sums2)
