"""Steps of one plan that switch between two weight sets.

Each switch makes ``qmuon_step`` rebuild the plan's Newton-Schulz tables
(problem descriptors, tensor maps, tile lists).  The steps are enqueued on a
non-blocking stream with no host synchronisation in between, so the host
rebuilds the tables for step t+1 while step t still runs on the GPU.  The
rebuilt tables must reach the GPU in stream order, so every weight set,
the q8 state, the absmax, the U left in the gradient buffers and the group
sums must equal, bit for bit, those of the same steps run with the host
waiting for each step before the next.  The two runs start from identical
seeded inputs, so the test also pins that a step is deterministic.
"""

import math

import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads

from gpu_util import random_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)


def _weights(mats, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return [(torch.randn(m.rows, m.cols, generator=g, device="cuda") * 0.02).contiguous() for m in mats]


def _run(shapes, tile, P, steps, wait_each):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    states = [workloads.random_state(m, 700 + i, device="cuda") for i, m in enumerate(mats)]
    wsets = [_weights(mats, 710), _weights(mats, 720)]
    grads = [[random_grad(m.numel, "bf16", 730 + 10 * t + i).reshape(m.rows, m.cols) for i, m in enumerate(mats)]
             for t in range(steps)]
    bufs = [torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device="cuda") for m in mats]
    plan = q.qmuon_plan_create([(s[0], s[1], b, m.rows, m.cols) for s, b, m in zip(states, bufs, mats)],
                               "int8", "bf16", tile=tile)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    info = q.qmuon_plan_info(plan)
    sums = torch.zeros(steps, max(info["n_full_groups"], info["n_block_groups"]), device="cuda")
    eta_block = 0.02 / math.sqrt(tile[0] * tile[1])
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for t in range(1, steps + 1):
            for b, g in zip(bufs, grads[t - 1]):
                b.copy_(g)
            q.qmuon_step(plan, t, P, 0.95, 0.02, eta_block, wsets[(t - 1) % 2], COEFFS, 5, sums[t - 1], ws,
                         stream=stream)
            if wait_each:
                stream.synchronize()
    q.qmuon_sync_status(ws, stream=stream)
    torch.cuda.synchronize()
    return {"q8": [s[0] for s in states], "absmax": [s[1] for s in states], "w0": wsets[0], "w1": wsets[1],
            "U": bufs, "sums": [sums]}


@pytest.mark.parametrize("shapes,tile,P", [
    ([(2048, 4096), (1024, 2048)], (1, 1), 1),     # every step full: the full-step tables switch
    ([(2048, 4096), (1024, 2048)], (1, 2), 0),     # every step a block step: the block tables switch
])
def test_switching_weights_rebuilds_tables_in_stream_order(shapes, tile, P):
    ran_ahead = _run(shapes, tile, P, 4, wait_each=False)
    waited = _run(shapes, tile, P, 4, wait_each=True)
    for key, got in ran_ahead.items():
        for i, (a, b) in enumerate(zip(got, waited[key])):
            assert torch.equal(a, b), f"{key}[{i}] differs when the host runs ahead"
