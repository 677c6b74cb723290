"""The non-finite counter: blocks whose momentum holds a NaN or an infinity
are counted, through the update entry and through qmuon_step; finite inputs
count nothing."""

import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads

from gpu_util import random_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)


def _case():
    shapes = [(64, 512), (37, 96), (256, 256)]
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    states = [workloads.random_state(m, 3 + i, device="cuda") for i, m in enumerate(mats)]
    grads = [random_grad(m.numel, "bf16", 9 + i).reshape(m.rows, m.cols) for i, m in enumerate(mats)]
    return mats, states, grads


def test_counter_counts_nonfinite_blocks():
    mats, states, grads = _case()
    flat = [g.view(-1) for g in grads]
    flat[0][3 * 256 + 17] = float("nan")      # block 3 of tensor 0
    flat[0][3 * 256 + 200] = float("inf")     # the same block again: counted once
    flat[0][7 * 256] = float("-inf")          # block 7
    flat[1][3400] = float("nan")              # the last, partial block of tensor 1 (37 x 96 = 13 blocks + 224)
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, mats)], "int8", "bf16")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.qmuon_plan_set_nonfinite_counter(plan, cnt)
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, 0.9, 0, None, None, ws)
    q.qmuon_sync_status(ws)
    assert int(cnt.item()) == 3
    # detached: nothing more is counted
    q.qmuon_plan_set_nonfinite_counter(plan, None)
    q.qmuon_update_multi_normalize_groups(plan, 0.9, 0, None, None, ws)
    q.qmuon_sync_status(ws)
    assert int(cnt.item()) == 3


def test_counter_through_the_step_and_finite_inputs():
    mats, states, grads = _case()
    weights = [torch.zeros(m.rows, m.cols, device="cuda") for m in mats]
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, mats)], "int8", "bf16")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.qmuon_plan_set_nonfinite_counter(plan, cnt)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    sums = torch.zeros(len(mats), device="cuda")
    q.qmuon_step(plan, 1, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, sums, ws)
    q.qmuon_sync_status(ws)
    assert int(cnt.item()) == 0
    grads[2].view(-1)[100] = float("nan")
    q.qmuon_step(plan, 2, 1, 0.9, 0.02, 0.02, weights, COEFFS, 5, sums, ws)
    q.qmuon_sync_status(ws)
    assert int(cnt.item()) == 1


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("sr", [False, True], ids=["nearest", "stochastic"])
def test_nonfinite_blocks_follow_the_oracle(q8_kind, sr):
    # Blocks with a NaN or an infinity in the momentum still follow the
    # oracle's rules bit for bit: NaN lanes are ignored by the absmax, a NaN
    # product is quantised to 0 and an infinite absmax gives zero codes.  The
    # stored momentum matches on every element that is not NaN (a NaN is
    # stored as some NaN).
    import numpy as np
    from oracle import codec
    from gpu_util import to_oracle_grad

    shapes = [(64, 512), (37, 96)]
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    states = [workloads.random_state(m, 30 + i, q8_kind, device="cuda") for i, m in enumerate(mats)]
    grads = [random_grad(m.numel, "bf16", 90 + i).reshape(m.rows, m.cols) for i, m in enumerate(mats)]
    flat = [g.view(-1) for g in grads]
    flat[0][3 * 256 + 17] = float("nan")      # a NaN among finite values
    flat[0][5 * 256 + 200] = float("inf")     # an infinity: absmax inf, every code 0
    flat[0][7 * 256] = float("-inf")
    flat[0][9 * 256:10 * 256] = float("nan")  # a block of NaN only: absmax 0
    flat[1][3400] = float("nan")              # the partial last block of the second tensor
    host = [(s.cpu().numpy().copy(), a.cpu().numpy().copy(), to_oracle_grad(g, "bf16")) for (s, a), g in
            zip(states, grads)]
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states, grads, mats)],
                               q8_kind, "bf16")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    if sr:
        q.qmuon_update_multi_normalize_groups_sr(plan, 0.9, 0, 1234, 3, None, None, ws)
    else:
        q.qmuon_update_multi_normalize_groups(plan, 0.9, 0, None, None, ws)
    q.qmuon_sync_status(ws)
    res, _, _, _ = codec.multi_update([h[0] for h in host], [h[1] for h in host], [h[2] for h in host], 0.9,
                                      q8_kind=q8_kind, sr_seed=1234 if sr else None, sr_step=3)
    for i, ((s, a), r) in enumerate(zip(states, res)):
        np.testing.assert_array_equal(s.cpu().numpy(), r.q8, err_msg=str(i))
        np.testing.assert_array_equal(a.cpu().numpy(), r.absmax, err_msg=str(i))
        got = to_oracle_grad(grads[i], "bf16")
        nan = np.isnan(codec.f32_from_bf16_bits(r.grad))
        assert np.isnan(codec.f32_from_bf16_bits(got[nan])).all()
        np.testing.assert_array_equal(got[~nan], r.grad[~nan], err_msg=str(i))
    assert res[0].absmax[5] == np.inf and res[0].absmax[9] == 0.0   # the cases are really there
