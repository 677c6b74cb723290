"""Guard bytes around every buffer each entry writes (an out-of-bounds write
shows up as a changed guard byte): the update in all its modes and with
stochastic requantisation, the multi-tensor carrier, Newton-Schulz on strided
matrices (the columns between cols and the row stride are guards too) and fed
from an MXFP8 carrier (which it only reads), the
MuonBP step on ragged shapes, the allocation-free update and the GRASP step.
Shapes are chosen for ragged tails: sizes that are no multiple of 256, 32, the
64 x 64 TMA box or the 256 x 256 tile."""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import grasp

from gpu_util import Guarded, random_grad

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)
RAGGED = [(37, 96), (300, 1024), (1, 32), (129, 200), (257, 64)]
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _state(m, seed, q8_kind):
    qs, a = workloads.random_state(m, seed, q8_kind, device="cuda")
    gq, ga = Guarded(qs.shape, qs.dtype), Guarded(a.shape, a.dtype)
    gq.t.copy_(qs)
    ga.t.copy_(a)
    return gq, ga


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
@pytest.mark.parametrize("grad_dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", [0, 1, 2, "sr"])
def test_update_writes_stay_in_bounds(q8_kind, grad_dtype, mode):
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(RAGGED)]
    st = [_state(m, 10 + i, q8_kind) for i, m in enumerate(mats)]
    gr = []
    for i, m in enumerate(mats):
        g = Guarded((m.numel,), DT[grad_dtype])
        g.t.copy_(random_grad(m.numel, grad_dtype, 20 + i))
        gr.append(g)
    plan = q.qmuon_plan_create([(s[0].t, s[1].t, g.t, m.rows, m.cols) for s, g, m in zip(st, gr, mats)],
                               q8_kind, grad_dtype)
    sums, inv = Guarded((len(mats),), torch.float32), Guarded((len(mats),), torch.float32)
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    if mode == "sr":
        q.qmuon_update_multi_normalize_groups_sr(plan, 0.9, 2, 7, 3, sums.t, inv.t, ws)
    else:
        q.qmuon_update_multi_normalize_groups(plan, 0.9, mode, sums.t, inv.t, ws)
    q.qmuon_sync_status(ws)
    for b in [x for s in st for x in s] + gr + [sums, inv]:
        b.check((q8_kind, grad_dtype, mode))


def test_carrier_multi_writes_stay_in_bounds():
    shapes = [(37, 96), (300, 1024), (1, 32), (129, 224)]
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    st = [_state(m, 30 + i, "int8") for i, m in enumerate(mats)]
    gr = []
    for i, m in enumerate(mats):
        g = Guarded((m.numel,), torch.bfloat16)
        g.t.copy_(random_grad(m.numel, "bf16", 40 + i))
        gr.append(g)
    plan = q.qmuon_plan_create([(s[0].t, s[1].t, g.t, m.rows, m.cols) for s, g, m in zip(st, gr, mats)], "int8", "bf16")
    pay = [Guarded((m.numel,), torch.uint8) for m in mats]
    sca = [Guarded((m.rows * (m.cols // 32),), torch.uint8) for m in mats]
    inv, sums = Guarded((len(mats),), torch.float32), Guarded((len(mats),), torch.float32)
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier_multi(plan, 0.9, [p.t for p in pay], [s.t for s in sca], inv.t, ws, group_sumsq=sums.t)
    q.qmuon_sync_status(ws)
    for b in [x for s in st for x in s] + gr + pay + sca + [inv, sums]:
        b.check("carrier")


@pytest.mark.parametrize("shape,ld", [((96, 160), 168), ((300, 520), 528), ((520, 136), 200), ((8, 16), 24),
                                      ((1000, 264), 264)])
def test_newton_schulz_strided_stays_in_bounds(shape, ld):
    rows, cols = shape
    buf = Guarded((rows, ld), torch.bfloat16)
    gap = torch.full((rows, ld - cols), 1234.0, dtype=torch.bfloat16, device="cuda")
    buf.t[:, cols:] = gap
    x = buf.t[:, :cols]
    x.copy_((torch.randn(rows, cols, device="cuda") / (rows * cols) ** 0.5).to(torch.bfloat16))
    prob = q.ns_problem(x, rows, cols, ld=ld)
    ws = torch.empty(q.qmuon_ns_workspace_size([prob]), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched([prob], 5, COEFFS, ws)
    q.qmuon_sync_status(ws)
    buf.check(shape)
    assert torch.equal(buf.t[:, cols:], gap), "columns between cols and the row stride were written"
    assert bool(torch.isfinite(x.float()).all())


@pytest.mark.parametrize("shape,ld", [((37, 96), 104), ((300, 544), 552), ((520, 160), 168), ((129, 224), 224)])
def test_newton_schulz_from_carrier_stays_in_bounds(shape, ld):
    # the carrier is only read (payload and scales unchanged, guards intact);
    # the output goes to x alone, whose row-stride gap survives
    rows, cols = shape
    m = workloads.Matrix("t", rows, cols)
    qs, a = workloads.zero_state(m, "int8", device="cuda")
    g = random_grad(m.numel, "bf16", 77)
    pay = Guarded((m.numel,), torch.uint8)
    sca = Guarded((rows * (cols // 32),), torch.uint8)
    inv = torch.zeros(1, device="cuda")
    ws = torch.empty(q.qmuon_carrier_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier(qs, a, g, rows, cols, "int8", "bf16", 0.9, pay.t, sca.t, inv, ws)
    torch.cuda.synchronize()
    pay_before, sca_before = pay.t.clone(), sca.t.clone()
    buf = Guarded((rows, ld), torch.bfloat16)
    gap = torch.full((rows, ld - cols), 1234.0, dtype=torch.bfloat16, device="cuda")
    buf.t[:, cols:] = gap
    x = buf.t[:, :cols]
    prob = q.ns_problem(x, rows, cols, ld=ld, inv_norm=inv, input_kind=q.QMUON_NS_MXFP8, payload=pay.t,
                        scale_inv=sca.t)
    ws2 = torch.empty(q.qmuon_ns_workspace_size([prob]), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched([prob], 5, COEFFS, ws2)
    q.qmuon_sync_status(ws2)
    for b in (buf, pay, sca):
        b.check(shape)
    assert torch.equal(pay.t, pay_before) and torch.equal(sca.t, sca_before)
    assert torch.equal(buf.t[:, cols:], gap), "columns between cols and the row stride were written"
    assert bool(torch.isfinite(x.float()).all())


@pytest.mark.parametrize("tile,P", [((1, 1), 1), ((2, 1), 0), ((1, 2), 2)])
def test_step_writes_stay_in_bounds(tile, P):
    shapes = [(300, 520), (520, 136), (8, 16), (130, 136)] if tile == (1, 1) else [(512, 512), (256, 1024), (64, 512)]
    mats = [workloads.Matrix(f"m{i}", r, c) for i, (r, c) in enumerate(shapes)]
    st = [_state(m, 50 + i, "int8") for i, m in enumerate(mats)]
    gr, wt = [], []
    for i, m in enumerate(mats):
        g = Guarded((m.rows, m.cols), torch.bfloat16)
        g.t.copy_(random_grad(m.numel, "bf16", 60 + i).reshape(m.rows, m.cols))
        gr.append(g)
        w = Guarded((m.rows, m.cols), torch.float32)
        w.t.copy_(torch.randn(m.rows, m.cols, device="cuda") * 0.02)
        wt.append(w)
    plan = q.qmuon_plan_create([(s[0].t, s[1].t, g.t, m.rows, m.cols) for s, g, m in zip(st, gr, mats)],
                               "int8", "bf16", tile=tile)
    info = q.qmuon_plan_info(plan)
    sums = Guarded((max(info["n_full_groups"], info["n_block_groups"]),), torch.float32)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    for t in (1, 2):
        q.qmuon_step(plan, t, P, 0.95, 0.02, 0.01, [w.t for w in wt], COEFFS, 5, sums.t, ws)
        q.qmuon_sync_status(ws)
    for b in [x for s in st for x in s] + gr + wt + [sums]:
        b.check((tile, P))


def test_noalloc_update_stays_in_bounds():
    m = workloads.Matrix("t", 129, 200)
    qs, a = _state(m, 70, "int8")
    g = Guarded((m.numel,), torch.bfloat16)
    g.t.copy_(random_grad(m.numel, "bf16", 71))
    s, inv = Guarded((1,), torch.float32), Guarded((1,), torch.float32)
    q.qmuon_update_normalize_noalloc(qs.t, a.t, g.t, m.rows, m.cols, "int8", "bf16", 0.9, s.t, inv.t)
    torch.cuda.synchronize()
    for b in (qs, a, g, s, inv):
        b.check("noalloc")


def test_grasp_writes_stay_in_bounds():
    shapes = [(201, 192), (9, 64), (1000, 128)]
    descs, bufs = [], []
    for i, (rows, cols) in enumerate(shapes):
        st = grasp.initial_state(rows, cols, np.random.default_rng(80 + i).standard_normal((cols, 8)).astype(np.float32))
        d = {}
        for k in ("res", "res_rmax", "res_cmax", "p", "p_rmax", "p_cmax", "r", "r_rmax", "r_cmax"):
            a = np.ascontiguousarray(getattr(st, k))
            gb = Guarded(a.shape, torch.from_numpy(a).dtype)
            gb.t.copy_(torch.from_numpy(a))
            d[k] = gb
        g = Guarded((rows, cols), torch.bfloat16)
        g.t.copy_(random_grad(rows * cols, "bf16", 90 + i).reshape(rows, cols))
        d["grad"] = g
        bufs += list(d.values())
        descs.append(q.grasp_matrix(rows, cols, *[d[k].t for k in ("res", "res_rmax", "res_cmax", "p", "p_rmax",
                                                                   "p_cmax", "r", "r_rmax", "r_cmax", "grad")]))
    ws = torch.empty(q.qmuon_grasp_workspace_size(descs), dtype=torch.uint8, device="cuda")
    q.qmuon_grasp_step(descs, 0.9, ws)
    q.qmuon_sync_status(ws)
    for b in bufs:
        b.check("grasp")
