"""MuonBP steps captured into a CUDA graph and replayed.

Once a plan's Newton-Schulz tables exist (qmuon_step_prepare), a step is a
workspace memset and a fixed sequence of launches whose arguments depend only
on the step index.  A training loop can therefore capture one period of P
steps (P - 1 block steps and a full step), each preceded by the copy of that
step's gradients into the plan's buffers, and replay it period after period.
The replays must leave the q8 state, absmax, fp32 weights and the update U
(in the gradient buffers) bit-identical to the same steps run eagerly.
"""

import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads

pytestmark = pytest.mark.gpu

COEFFS = workloads.COEFFS
P = 3
SHAPES = [(256, 1024), (1024, 512), (512, 512)]   # wide, tall and square on a 1 x 2 tiling (tile rows of whole 256-element blocks)


def _setup(seed_state):
    torch.manual_seed(seed_state)
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(SHAPES)]
    states = [workloads.random_state(m, 100 + i, device="cuda") for i, m in enumerate(mats)]
    grads = [torch.zeros(m.rows, m.cols, dtype=torch.bfloat16, device="cuda") for m in mats]
    weights = [(torch.randn(m.rows, m.cols, device="cuda", generator=torch.Generator("cuda").manual_seed(200 + i))
                * 0.02).contiguous() for i, m in enumerate(mats)]
    plan = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                               "int8", "bf16", tile=(1, 2))
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    info = q.qmuon_plan_info(plan)
    sums = torch.zeros(max(info["n_block_groups"], info["n_full_groups"]), device="cuda")
    q.qmuon_step_prepare(plan, weights, ws)
    return dict(mats=mats, states=states, grads=grads, weights=weights, plan=plan, ws=ws, sums=sums)


def _step(S, t, src):
    for g, s in zip(S["grads"], src):
        g.copy_(s)
    q.qmuon_step(S["plan"], t, P, 0.95, 0.02, 0.01, S["weights"], COEFFS, 5, S["sums"], S["ws"])


def _same(A, B, what):
    # byte-level equality of every output the steps write
    for i in range(len(SHAPES)):
        pairs = (("q8", A["states"][i][0], B["states"][i][0]), ("absmax", A["states"][i][1], B["states"][i][1]),
                 ("weights", A["weights"][i], B["weights"][i]), ("U", A["grads"][i], B["grads"][i]))
        for name, a, b in pairs:
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (what, i, name)


def test_captured_period_replays_like_eager_steps():
    # each period's gradients: one fresh batch per step of the period
    gen = torch.Generator("cuda").manual_seed(7)
    src = [[(torch.randn(r, c, device="cuda", generator=gen) * 1e-2).to(torch.bfloat16) for r, c in SHAPES]
           for _ in range(P)]
    A = _setup(1)   # eager
    B = _setup(1)   # graph
    _same(A, B, "initial")
    for t in range(1, P + 1):
        _step(A, t, src[t - 1])
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=stream):
        for t in range(1, P + 1):
            _step(B, t, src[t - 1])
    torch.cuda.current_stream().wait_stream(stream)
    # capturing ran nothing: B is still at its initial state
    g.replay()
    torch.cuda.synchronize()
    q.qmuon_sync_status(B["ws"])
    _same(A, B, "first period")

    # the next period (t = P + 1 .. 2P has the same block / full pattern)
    for t in range(P + 1, 2 * P + 1):
        _step(A, t, src[t - P - 1])
    g.replay()
    torch.cuda.synchronize()
    q.qmuon_sync_status(A["ws"])
    q.qmuon_sync_status(B["ws"])
    _same(A, B, "second period")
