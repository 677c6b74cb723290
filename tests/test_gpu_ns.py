"""GPU parity of the Newton-Schulz engine (tcgen05) and of the MuonBP step.

Single-iteration runs with one coefficient switched on at a time check each
term of the three tensor-core products on its own (wide and tall operands,
ragged shapes) against fp64 products of the same bf16-rounded intermediates
(the a X term travels on the diagonal of the bf16 polynomial B); the
five-iteration runs and the steps are held to the oracle tolerance:
relative Frobenius error <= 2e-2 and per-row cosine >= 0.999.
"""

import math

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import codec, muonbp, ns

from gpu_util import bf16_to_f64, min_row_cos, one_iteration_reference, random_grad, rel_fro, to_oracle_grad

pytestmark = pytest.mark.gpu

COEFFS = workloads.COEFFS


def _run_ns(mats, iters, coeffs, invs=None):
    probs = []
    for i, Mt in enumerate(mats):
        r, c = Mt.shape
        probs.append(q.ns_problem(Mt, r, c, inv_norm=None if invs is None else invs[i]))
    ws = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, iters, coeffs, ws)
    q.qmuon_sync_status(ws)


SHAPES = [(128, 256), (256, 128), (8, 16), (24, 40), (40, 24), (300, 520), (520, 304), (512, 512), (1000, 136),
          (64, 1024)]


@pytest.mark.parametrize("coeffs", [(1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0), COEFFS])
def test_single_iteration_products(coeffs):
    rng = np.random.default_rng(1)
    mats, ref = [], []
    for r, c in SHAPES:
        M = rng.standard_normal((r, c)).astype(np.float32)
        Mt = torch.from_numpy(M).to(torch.bfloat16).cuda()
        Mb = Mt.float().cpu().numpy().astype(np.float64)
        inv = 1.0 / np.linalg.norm(Mb)
        mats.append(Mt)
        ref.append(one_iteration_reference(Mb, coeffs, inv))
    invs = [torch.tensor([1.0 / np.linalg.norm(bf16_to_f64(m))], dtype=torch.float32, device="cuda") for m in mats]
    _run_ns(mats, 1, coeffs, invs)
    for (r, c), Mt, R in zip(SHAPES, mats, ref):
        got = bf16_to_f64(Mt)
        err = rel_fro(got, R)
        assert err <= 6e-3, ((r, c), coeffs, err)


@pytest.mark.parametrize("shape", SHAPES + [(2048, 1024), (1024, 3072)])
def test_five_iterations_vs_oracle(shape):
    r, c = shape
    g = random_grad(r * c, "bf16", 77).reshape(r, c)
    M = bf16_to_f64(g)
    inv_h = 1.0 / (np.linalg.norm(M) + 1e-7)
    inv = torch.tensor([inv_h], dtype=torch.float32, device="cuda")
    ref = ns.newton_schulz(M, inv_norm=float(inv.item()))
    _run_ns([g], 5, COEFFS, [inv])
    got = bf16_to_f64(g)
    assert rel_fro(got, ref) <= 2e-2
    assert min_row_cos(got, ref) >= 0.999


def test_symmetric_products_read_only_their_upper_tiles():
    # The Gram A and the polynomial B hold only their 256 x 256 tiles on or
    # above the diagonal; the products that read them take the blocks below
    # it transposed from above.  With every workspace byte set to 0xFF
    # (a bf16 NaN) before the call, any read of a block that was never
    # written would put NaNs into X.  Shapes with two to eight row tiles,
    # wide and tall, ragged and exact, in one batch.
    shapes = [(300, 520), (520, 304), (512, 2048), (2048, 1024), (1100, 1536)]
    mats, refs, invs = [], [], []
    for i, (r, c) in enumerate(shapes):
        g = random_grad(r * c, "bf16", 90 + i).reshape(r, c)
        M = bf16_to_f64(g)
        inv = torch.tensor([1.0 / (np.linalg.norm(M) + 1e-7)], dtype=torch.float32, device="cuda")
        refs.append(ns.newton_schulz(M, inv_norm=float(inv.item())))
        mats.append(g)
        invs.append(inv)
    probs = [q.ns_problem(g, g.shape[0], g.shape[1], inv_norm=inv) for g, inv in zip(mats, invs)]
    ws = torch.full((q.qmuon_ns_workspace_size(probs),), 0xFF, dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, 5, COEFFS, ws)
    q.qmuon_sync_status(ws)
    for shape, g, ref in zip(shapes, mats, refs):
        got = bf16_to_f64(g)
        assert np.isfinite(got).all(), shape
        assert rel_fro(got, ref) <= 2e-2, shape
        assert min_row_cos(got, ref) >= 0.999, shape


def test_batch_of_mixed_problems_and_strided_view():
    # one launch sequence over problems of different shapes, one of them a
    # column block of a wider matrix (row stride larger than its width)
    base = random_grad(384 * 1024, "bf16", 5).reshape(384, 1024)
    view_ref = bf16_to_f64(base[:, 256:512])
    others = [random_grad(r * c, "bf16", 6 + i).reshape(r, c) for i, (r, c) in enumerate([(96, 200), (700, 256)])]
    inputs = [view_ref] + [bf16_to_f64(t) for t in others]
    # the inverse norms travel as device scalars (a NULL inverse norm means 1)
    invs = [torch.tensor([1.0 / (np.linalg.norm(x) + 1e-7)], dtype=torch.float32, device="cuda") for x in inputs]
    refs = [ns.newton_schulz(x, inv_norm=float(i.item())) for x, i in zip(inputs, invs)]
    untouched = base[:, :256].clone()
    probs = [q.ns_problem(base.data_ptr() + 256 * 2, 384, 256, ld=1024, inv_norm=invs[0])] + \
            [q.ns_problem(t, t.shape[0], t.shape[1], inv_norm=i) for t, i in zip(others, invs[1:])]
    ws = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, 5, COEFFS, ws)
    q.qmuon_sync_status(ws)
    outs = [bf16_to_f64(base[:, 256:512])] + [bf16_to_f64(t) for t in others]
    for got, ref in zip(outs, refs):
        assert rel_fro(got, ref) <= 2e-2 and min_row_cos(got, ref) >= 0.999
    assert torch.equal(base[:, :256], untouched)


def _step_case(shapes, tile, seed):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    dev = "cuda"
    states_d, weights_d, grads_d = [], [], []
    for i, m in enumerate(mats):
        qs, a = workloads.random_state(m, seed + i, device=dev)
        states_d.append((qs, a))
        weights_d.append((torch.randn(m.rows, m.cols, device=dev) * 0.02).contiguous())
        grads_d.append(torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device=dev))
    plan = q.qmuon_plan_create([(s, a, g, m.rows, m.cols) for (s, a), g, m in zip(states_d, grads_d, mats)],
                               "int8", "bf16", tile=tile)
    host = [muonbp.MatrixState(m.rows, m.cols, s.cpu().numpy(), a.cpu().numpy(), w.cpu().numpy())
            for (s, a), w, m in zip(states_d, weights_d, mats)]
    return mats, plan, states_d, weights_d, grads_d, host


def _run_steps(shapes, tile, P, steps, seed):
    mats, plan, states_d, weights_d, grads_d, host = _step_case(shapes, tile, seed)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    eta_full, eta_block = 0.02, 0.02 / math.sqrt(tile[0] * tile[1])
    for t in range(1, steps + 1):
        gh = []
        for i, (m, g) in enumerate(zip(mats, grads_d)):
            src = random_grad(m.numel, "bf16", 900 + 10 * t + i).reshape(m.rows, m.cols)
            g.copy_(src)
            gh.append(to_oracle_grad(g, "bf16"))
        full = muonbp.is_full_step(t, P)
        ngr = q.qmuon_plan_info(plan)["n_full_groups" if full else "n_block_groups"]
        sums = torch.zeros(ngr, device="cuda")
        w_before = [w.cpu().numpy().astype(np.float64) for w in weights_d]
        q.qmuon_step(plan, t, P, 0.95, eta_full, eta_block, weights_d, COEFFS, 5, sums, ws)
        q.qmuon_sync_status(ws)
        host, U, info = muonbp.muonbp_step(t, P, host, gh, 0.95, eta_full, eta_block, tile=tile)
        assert info["full"] == full
        np.testing.assert_allclose(sums.cpu().numpy(), info["S"], rtol=1e-5)
        for i, m in enumerate(mats):
            np.testing.assert_array_equal(states_d[i][0].cpu().numpy(), host[i].q8)
            np.testing.assert_array_equal(states_d[i][1].cpu().numpy(), host[i].absmax)
            got = bf16_to_f64(grads_d[i])
            ref = codec.f32_from_bf16_bits(U[i]).astype(np.float64)
            th, tw = (m.rows, m.cols) if full else (m.rows // tile[0], m.cols // tile[1])
            for bi in range(m.rows // th):
                for bj in range(m.cols // tw):
                    sl = (slice(bi * th, (bi + 1) * th), slice(bj * tw, (bj + 1) * tw))
                    assert rel_fro(got[sl], ref[sl]) <= 2e-2 and min_row_cos(got[sl], ref[sl]) >= 0.999, (t, m, bi, bj)
            # the weight moved by eta * U (eta_full on full steps, eta_block
            # otherwise): compare the applied updates, and check that every
            # weight moved by exactly fl(eta * bf16(U)) of the U left in place
            w_after = weights_d[i].cpu().numpy()
            dW = w_after.astype(np.float64) - w_before[i]
            dW_ref = host[i].weight.astype(np.float64) - w_before[i]
            assert rel_fro(dW, dW_ref) <= 2e-2, (t, m)
            eta = np.float32(eta_full if full else eta_block)
            u32 = grads_d[i].float().cpu().numpy()
            expect = (w_before[i].astype(np.float32) - (eta * u32).astype(np.float32)).astype(np.float32)
            np.testing.assert_array_equal(w_after, expect)
        # keep both sides on the same weights so errors do not accumulate
        for i in range(len(mats)):
            weights_d[i].copy_(torch.from_numpy(host[i].weight).cuda())


@pytest.mark.parametrize("P", [5, 1, 0])
def test_muonbp_steps_vs_oracle(P):
    _run_steps([(512, 2048), (256, 2048), (1024, 4096), (2048, 2048)], (1, 8), P, 5, 40)


def test_steps_ragged_shapes():
    # full steps on shapes that are not multiples of the 256 x 256 tile (wide,
    # tall, tiny): partial weight and output boxes at every edge
    _run_steps([(300, 520), (520, 136), (8, 16), (1000, 264), (130, 136)], (1, 1), 1, 2, 70)


def test_steps_row_tiles():
    # block steps on a 2 x 1 row tiling: problems that start mid-matrix
    _run_steps([(512, 136), (1024, 256)], (2, 1), 0, 2, 90)


def test_steps_long_k():
    # full steps whose update tiles have K >= 2048 on average: the weight pass
    # with the one-step weight ring and five operand stages (a ragged shape too)
    _run_steps([(2048, 2304), (2100, 2056)], (1, 1), 1, 2, 110)


@pytest.mark.parametrize("P,t", [(2, 1), (2, 2)])
def test_step_results_do_not_depend_on_workspace_contents(P, t):
    # a block step (t = 1) and a full step (t = 2) with every workspace byte
    # set to 0xFF (bf16 NaN) before the call give bit-for-bit the outputs of
    # the same step with a zeroed workspace: nothing reads a byte of the
    # workspace that the call did not write first (the symmetric matrices'
    # blocks below the diagonal among them)
    shapes = [(512, 2048), (1100, 1536), (1024, 512)]
    tile = (1, 2)
    out = []
    for fill in (0x00, 0xFF):
        mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
        states = [workloads.random_state(m, 120 + i, device="cuda") for i, m in enumerate(mats)]
        grads = [random_grad(m.numel, "bf16", 130 + i).reshape(m.rows, m.cols) for i, m in enumerate(mats)]
        weights = [(torch.randn(m.rows, m.cols, device="cuda", generator=torch.Generator("cuda").manual_seed(140 + i))
                    * 0.02).contiguous() for i, m in enumerate(mats)]
        plan = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                                   "int8", "bf16", tile=tile)
        ws = torch.full((q.qmuon_workspace_size(plan, q.QMUON_WS_STEP),), fill, dtype=torch.uint8, device="cuda")
        info = q.qmuon_plan_info(plan)
        sums = torch.zeros(max(info["n_block_groups"], info["n_full_groups"]), device="cuda")
        q.qmuon_step(plan, t, P, 0.95, 0.02, 0.01, weights, COEFFS, 5, sums, ws)
        q.qmuon_sync_status(ws)
        out.append([x.clone() for s in states for x in s] + [g.clone() for g in grads] +
                   [w.clone() for w in weights] + [sums.clone()])
    for a, b in zip(*out):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
