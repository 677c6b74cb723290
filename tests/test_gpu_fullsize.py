"""GPU parity at the synthetic workloads' full sizes, launched the way the
benchmark launches them.

The oracle cannot afford whole 0.5-0.9 G-parameter workloads, so each check
takes what it can compute one by one or whole-but-affordable:

* sampled 256-element quantization blocks of every matrix: codes, absmax and
  (before Newton-Schulz overwrites it) the stored momentum, bit-exact against
  ``oracle.codec.momentum_update`` run on those blocks alone (the codec is
  blockwise independent);
* whole matrices or tiles the fp64 oracle orthogonalises in seconds: group
  sums (rtol 1e-5) and the Newton-Schulz output (relative Frobenius 2e-2,
  per-row cosine 0.999 for bf16 inputs; 5e-2 / 0.995 for the MXFP8 carrier);
* every master weight of the MuonBP step: ``W_after == fl(W_before -
  fl(eta * U))`` exactly, with ``U`` the bf16 update left in the gradient
  buffer -- a property that holds at any size.

Workloads: the single 512 x 512 matrix (its three steps), the fused-QKV + MLP grouped set (3 row groups of a 12288 x 4096
tensor + 8 MLP matrices), MuonBP on four Llama-8B layers (1 x 8 column
tiles, P = 5; a block step and a full step), the MXFP8 carrier on the same
layers, and the 4-bit GRASP state of those 28 matrices in one call (sampled
64-row strips of M_t bit-exact, one whole 1024 x 4096 matrix against the
oracle's step).
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads
from oracle import carrier, codec, grasp, muonbp, ns

from gpu_util import bf16_to_f64, min_row_cos, rel_fro, to_oracle_grad

pytestmark = pytest.mark.gpu

BLK = 256


def _blocks_of(t: torch.Tensor, idx) -> np.ndarray:
    """Flat contents of the 256-element blocks ``idx`` of a block-multiple tensor."""
    sel = torch.as_tensor(np.asarray(idx), device=t.device, dtype=torch.long)
    return t.reshape(-1, BLK).index_select(0, sel).reshape(-1)


def _sample(mats, states, grads, rng, per):
    """Inputs of ``per`` random blocks of every matrix, copied before the call."""
    picks = []
    for i, m in enumerate(mats):
        assert m.numel % BLK == 0
        idx = np.sort(rng.choice(m.numel // BLK, size=per, replace=False))
        picks.append((i, idx, _blocks_of(states[i][0], idx).cpu().numpy(),
                      states[i][1][torch.as_tensor(idx, device=states[i][1].device)].cpu().numpy(),
                      to_oracle_grad(_blocks_of(grads[i], idx), "bf16")))
    return picks


def _check_sampled(picks, states, beta, q8_kind, grads=None):
    for i, idx, hq, ha, hg in picks:
        r = codec.momentum_update(hq, ha, hg, beta, q8_kind=q8_kind)
        np.testing.assert_array_equal(_blocks_of(states[i][0], idx).cpu().numpy(), r.q8, err_msg=str(i))
        np.testing.assert_array_equal(states[i][1][torch.as_tensor(idx, device=states[i][1].device)].cpu().numpy(),
                                      r.absmax, err_msg=str(i))
        if grads is not None:   # the stored momentum, while the buffer still holds it
            np.testing.assert_array_equal(to_oracle_grad(_blocks_of(grads[i], idx), "bf16"), r.grad, err_msg=str(i))


def _whole_input(states, grads, i):
    return states[i][0].cpu().numpy().copy(), states[i][1].cpu().numpy().copy(), to_oracle_grad(grads[i], "bf16")


def _assert_ns(got: np.ndarray, ref: np.ndarray, what, fro=2e-2, cos=0.999):
    e, c = rel_fro(got, ref), min_row_cos(got, ref)
    assert e <= fro and c >= cos, (what, e, c)


# ---------------------------------------------------------------------------
# grouped QKV + MLP: update with deferred group norms, then Newton-Schulz on
# the row-group slices
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_grouped_qkv_mlp_full_size(q8_kind):
    w = workloads.get(3, q8_kind=q8_kind)
    mats = w.matrices
    rng = np.random.default_rng(3)
    states = [workloads.random_state(m, 700 + i, w.q8_kind, device="cuda") for i, m in enumerate(mats)]
    grads = [workloads.make_grad(w, i, 1, device="cuda") for i in range(len(mats))]
    picks = _sample(mats, states, grads, rng, 32)
    whole = {0: _whole_input(states, grads, 0), 5: _whole_input(states, grads, 5)}   # qkv, mlp0.down

    segs = [(s.tensor_index, s.start, s.length, s.group_id) for s in w.segments]
    plan = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                               w.q8_kind, "bf16", segments=segs, n_groups=w.n_groups)
    sums = torch.zeros(w.n_groups, device="cuda")
    inv = torch.zeros(w.n_groups, device="cuda")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_multi_normalize_groups(plan, w.beta, 2, sums, inv, ws)
    q.qmuon_sync_status(ws)
    _check_sampled(picks, states, w.beta, w.q8_kind, grads)

    probs = [q.ns_problem(grads[t][r0:r0 + nr], nr, mats[t].cols, inv_norm=inv.data_ptr() + 4 * k)
             for k, (t, r0, nr) in enumerate(w.ns_slices)]
    ws_n = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n)
    q.qmuon_sync_status(ws_n)

    # the fused QKV tensor: its three row groups' sums, and the middle group's
    # orthogonalised slice (it starts 4096 rows into the tensor)
    r = codec.momentum_update(*whole[0], w.beta, q8_kind=w.q8_kind)
    third = mats[0].numel // 3
    S_ref = [float(np.sum(r.block_sumsq[g * third // BLK:(g + 1) * third // BLK])) for g in range(3)]
    np.testing.assert_allclose(sums[:3].cpu().numpy(), S_ref, rtol=1e-5)
    np.testing.assert_allclose(inv[:3].cpu().numpy(), 1.0 / (np.sqrt(S_ref) + codec.EPS), rtol=1e-5)
    M = codec.f32_from_bf16_bits(r.grad).reshape(mats[0].rows, mats[0].cols).astype(np.float64)
    _assert_ns(bf16_to_f64(grads[0][4096:8192]), ns.newton_schulz(M[4096:8192], inv_norm=float(inv[1].item())),
               "qkv.k")
    # a 4096 x 14336 MLP matrix: its own group (7), orthogonalised whole
    r = codec.momentum_update(*whole[5], w.beta, q8_kind=w.q8_kind)
    np.testing.assert_allclose(sums[7].item(), float(np.sum(r.block_sumsq)), rtol=1e-5)
    if q8_kind == "int8":   # the uint8 codes decode to the same momentum: one Newton-Schulz check serves both
        M = codec.f32_from_bf16_bits(r.grad).reshape(mats[5].rows, mats[5].cols).astype(np.float64)
        _assert_ns(bf16_to_f64(grads[5]), ns.newton_schulz(M, inv_norm=float(inv[7].item())), "mlp0.down")


# ---------------------------------------------------------------------------
# MuonBP on four Llama-8B layers: the benchmark's plan, workspace and call
# ---------------------------------------------------------------------------

def _muonbp_case(w):
    mats = w.matrices
    states = [workloads.random_state(m, 800 + i, w.q8_kind, device="cuda") for i, m in enumerate(mats)]
    weights = [workloads.make_weight(w, i, device="cuda") for i in range(len(mats))]
    grads = [workloads.make_grad(w, i, 1, device="cuda") for i in range(len(mats))]
    plan = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                               w.q8_kind, "bf16", tile=w.tile)
    info = q.qmuon_plan_info(plan)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    q.qmuon_step_prepare(plan, weights, ws)
    sums = torch.zeros(max(info["n_full_groups"], info["n_block_groups"]), device="cuda")
    return mats, states, weights, grads, plan, ws, sums


def _check_weight_relation(mats, w_before, weights, grads, eta):
    # every element of every master weight: W_after = fl(W_before - fl(eta * U))
    eta = np.float32(eta)
    for i in range(len(mats)):
        wb = w_before[i].cpu().numpy()
        u32 = grads[i].float().cpu().numpy()
        expect = (wb - (eta * u32).astype(np.float32)).astype(np.float32)
        np.testing.assert_array_equal(weights[i].cpu().numpy(), expect, err_msg=mats[i].name)


def _oracle_matrix_step(w, t, mats, i, whole, w_before):
    """The oracle's MuonBP step on matrix ``i`` alone (its groups are its own)."""
    hq, ha, hg = whole
    st = muonbp.MatrixState(mats[i].rows, mats[i].cols, hq, ha, w_before[i].cpu().numpy())
    new, U, info = muonbp.muonbp_step(t, w.P, [st], [hg], w.beta, w.eta_full, w.eta_block, tile=w.tile,
                                      iters=w.iters, coeffs=w.coeffs, q8_kind=w.q8_kind)
    return new[0], U[0], info


def test_single_512_three_steps_as_benchmarked():
    # the one-matrix 512 x 512 workload as the benchmark runs it: qmuon_step
    # with P = 1 from a zero state for its three steps, each step against the
    # oracle's: codes and absmax bit-exact, the group sum to 1e-5, U within the
    # Newton-Schulz tolerance, and every weight by the exact update relation
    w = workloads.get(1)
    m = w.matrices[0]
    qs, a = workloads.zero_state(m, w.q8_kind, device="cuda")
    weight = workloads.make_weight(w, 0, device="cuda")
    g = torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device="cuda")
    plan = q.qmuon_plan_create([(qs, a, g, m.rows, m.cols)], w.q8_kind, "bf16", tile=w.tile)
    ws = torch.empty(q.qmuon_workspace_size(plan, q.QMUON_WS_STEP), dtype=torch.uint8, device="cuda")
    sums = torch.zeros(1, device="cuda")
    st = muonbp.MatrixState(m.rows, m.cols, qs.cpu().numpy().copy(), a.cpu().numpy().copy(),
                            weight.cpu().numpy().copy())
    for t in range(1, w.steps + 1):
        g.copy_(workloads.make_grad(w, 0, t, device="cuda").reshape(m.rows, m.cols))
        hg = to_oracle_grad(g, "bf16")
        w_before = weight.clone()
        q.qmuon_step(plan, t, w.P, w.beta, w.eta_full, w.eta_block, [weight], w.coeffs, w.iters, sums, ws)
        q.qmuon_sync_status(ws)
        new, U, info = muonbp.muonbp_step(t, w.P, [st], [hg], w.beta, w.eta_full, w.eta_block, tile=w.tile,
                                          iters=w.iters, coeffs=w.coeffs, q8_kind=w.q8_kind)
        assert info["full"]
        np.testing.assert_array_equal(qs.cpu().numpy(), new[0].q8, err_msg=str(t))
        np.testing.assert_array_equal(a.cpu().numpy(), new[0].absmax, err_msg=str(t))
        np.testing.assert_allclose(sums.item(), info["S"][0], rtol=1e-5, err_msg=str(t))
        _assert_ns(bf16_to_f64(g), codec.f32_from_bf16_bits(U[0]).astype(np.float64), ("512x512", t))
        _check_weight_relation([m], [w_before], [weight], [g], w.eta_full)
        st = new[0]


@pytest.mark.parametrize("t", [1, 5], ids=["block_step", "full_step"])
def test_muonbp_llama8b_full_size(t):
    w = workloads.get(4)
    mats, states, weights, grads, plan, ws, sums = _muonbp_case(w)
    full = muonbp.is_full_step(t, w.P)
    tr, tc = w.tile
    rng = np.random.default_rng(40 + t)
    picks = _sample(mats, states, grads, rng, 24)
    # whole matrices the oracle steps alone: k and down of layer 0, plus
    # gate (block step: 14336 x 512 tiles) or q (full step: 4096 x 4096)
    checked = [1, 6] + ([4] if not full else [0])
    whole = {i: _whole_input(states, grads, i) for i in checked}
    w_before = [x.clone() for x in weights]

    q.qmuon_step(plan, t, w.P, w.beta, w.eta_full, w.eta_block, weights, w.coeffs, w.iters, sums, ws)
    q.qmuon_sync_status(ws)
    torch.cuda.synchronize()

    _check_sampled(picks, states, w.beta, w.q8_kind)
    _check_weight_relation(mats, w_before, weights, grads, w.eta_full if full else w.eta_block)

    for i in checked:
        m = mats[i]
        got = bf16_to_f64(grads[i])
        if i == 6 and not full:
            # 4096 x 14336 in 1 x 8 tiles: one 4096 x 1792 tile (j = 3) from its
            # own blocks, as one rank holding that shard would compute it
            hq, ha, hg = whole[i]
            tw, bpr = m.cols // tc, m.cols // BLK
            j = 3
            idx = (np.arange(m.rows)[:, None] * bpr + j * (tw // BLK) + np.arange(tw // BLK)[None, :]).reshape(-1)
            sel = (idx[:, None] * BLK + np.arange(BLK)[None, :]).reshape(-1)
            r = codec.momentum_update(hq[sel], ha[idx], hg[sel], w.beta, q8_kind=w.q8_kind)
            g = i * tr * tc + j
            S = float(np.sum(r.block_sumsq))
            np.testing.assert_allclose(sums[g].item(), S, rtol=1e-5)
            M = codec.f32_from_bf16_bits(r.grad).reshape(m.rows, tw).astype(np.float64)
            ref = ns.newton_schulz(M, inv_norm=float(1.0 / (np.sqrt(S) + codec.EPS)), iters=w.iters,
                                   coeffs=w.coeffs)
            _assert_ns(got[:, j * tw:(j + 1) * tw], ref, (m.name, j))
            continue
        new, U, info = _oracle_matrix_step(w, t, mats, i, whole[i], w_before)
        ng = info["n_groups"]
        base = i if full else i * tr * tc
        np.testing.assert_allclose(sums[base:base + ng].cpu().numpy(), info["S"], rtol=1e-5, err_msg=m.name)
        np.testing.assert_array_equal(states[i][0].cpu().numpy(), new.q8, err_msg=m.name)
        np.testing.assert_array_equal(states[i][1].cpu().numpy(), new.absmax, err_msg=m.name)
        ref = codec.f32_from_bf16_bits(U).astype(np.float64)
        th, tw = (m.rows, m.cols) if full else (m.rows // tr, m.cols // tc)
        for bi in range(m.rows // th):
            for bj in range(m.cols // tw):
                sl = (slice(bi * th, (bi + 1) * th), slice(bj * tw, (bj + 1) * tw))
                _assert_ns(got[sl], ref[sl], (m.name, bi, bj))


# ---------------------------------------------------------------------------
# MXFP8 carrier on four Llama-8B layers: one multi-tensor carrier launch, then
# Newton-Schulz fed by the carrier
# ---------------------------------------------------------------------------

def test_carrier_llama8b_full_size():
    w = workloads.get(5)
    mats = w.matrices
    rng = np.random.default_rng(5)
    states = [workloads.random_state(m, 900 + i, w.q8_kind, device="cuda") for i, m in enumerate(mats)]
    grads = [workloads.make_grad(w, i, 1, device="cuda") for i in range(len(mats))]
    outs = [torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device="cuda") for m in mats]
    payload = [torch.empty(m.numel, dtype=torch.uint8, device="cuda") for m in mats]
    scale = [torch.empty(m.rows * (m.cols // 32), dtype=torch.uint8, device="cuda") for m in mats]
    inv = torch.zeros(len(mats), dtype=torch.float32, device="cuda")
    # sampled whole rows of every matrix (a row is a whole number of blocks)
    rows = []
    for i, m in enumerate(mats):
        r_idx = np.sort(rng.choice(m.rows, size=6, replace=False))
        bpr = m.cols // BLK
        idx = (r_idx[:, None] * bpr + np.arange(bpr)[None, :]).reshape(-1)
        rows.append((i, r_idx, idx, _blocks_of(states[i][0], idx).cpu().numpy(),
                     states[i][1][torch.as_tensor(idx, device="cuda")].cpu().numpy(),
                     to_oracle_grad(_blocks_of(grads[i], idx), "bf16")))
    k_in = _whole_input(states, grads, 1)   # layer 0's k, 1024 x 4096, checked whole

    plan = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                               w.q8_kind, "bf16")
    ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
    q.qmuon_update_mxfp8_carrier_multi(plan, w.beta, payload, scale, inv, ws)
    q.qmuon_sync_status(ws)
    probs = [q.ns_problem(o, m.rows, m.cols, inv_norm=inv.data_ptr() + 4 * i, input_kind=q.QMUON_NS_MXFP8,
                          payload=payload[i], scale_inv=scale[i]) for i, (o, m) in enumerate(zip(outs, mats))]
    ws_n = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device="cuda")
    q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n)
    q.qmuon_sync_status(ws_n)

    for i, r_idx, idx, hq, ha, hg in rows:
        m = mats[i]
        r = carrier.carrier_update(hq, ha, hg, w.beta, len(r_idx), m.cols, q8_kind=w.q8_kind)
        np.testing.assert_array_equal(_blocks_of(states[i][0], idx).cpu().numpy(), r.q8, err_msg=m.name)
        np.testing.assert_array_equal(states[i][1][torch.as_tensor(idx, device="cuda")].cpu().numpy(), r.absmax,
                                      err_msg=m.name)
        np.testing.assert_array_equal(payload[i].reshape(m.rows, m.cols)[torch.as_tensor(r_idx, device="cuda")]
                                      .cpu().numpy(), r.payload, err_msg=m.name)
        np.testing.assert_array_equal(scale[i].reshape(m.rows, m.cols // 32)[torch.as_tensor(r_idx, device="cuda")]
                                      .cpu().numpy(), r.scale_inv, err_msg=m.name)

    m = mats[1]
    r = carrier.carrier_update(*k_in, w.beta, m.rows, m.cols, q8_kind=w.q8_kind)
    np.testing.assert_array_equal(payload[1].cpu().numpy().reshape(m.rows, m.cols), r.payload)
    np.testing.assert_array_equal(scale[1].cpu().numpy().reshape(m.rows, m.cols // 32), r.scale_inv)
    np.testing.assert_allclose(inv[1].item(), r.inv_norm, rtol=1e-5)
    ref = ns.newton_schulz(carrier.decode_rows(r.payload, r.scale_inv), inv_norm=float(inv[1].item()),
                           iters=w.iters, coeffs=w.coeffs)
    _assert_ns(bf16_to_f64(outs[1]), ref, m.name, fro=5e-2, cos=0.995)


# ---------------------------------------------------------------------------
# the 4-bit GRASP state on the same 28 matrices, all in one call
# ---------------------------------------------------------------------------

def _random_grasp_state(rows, cols, gen):
    """A valid, non-trivial state: random codes and positive maxima (seeded)."""
    nbr, nbc = (rows + 63) // 64, cols // 64
    u = lambda *sh: torch.rand(*sh, generator=gen, device="cuda") * 0.9 + 0.1
    return dict(res=torch.randint(0, 256, (rows, cols // 2), generator=gen, device="cuda", dtype=torch.int32).to(torch.uint8),
                res_rmax=u(nbc, rows) * 0.02, res_cmax=u(nbr, cols) * 0.02,
                p=torch.randint(-127, 128, (rows, 8), generator=gen, device="cuda", dtype=torch.int32).to(torch.int8),
                p_rmax=u(rows) * 0.05, p_cmax=u(nbr, 8) * 0.05,
                r=torch.randint(-127, 128, (cols, 8), generator=gen, device="cuda", dtype=torch.int32).to(torch.int8),
                r_rmax=u(cols), r_cmax=u((cols + 63) // 64, 8))


def _grasp_host(d):
    """The device state as the oracle holds it (the factors' row maxima as 1 x n)."""
    n = lambda k: d[k].cpu().numpy()
    return grasp.GraspState(res=n("res"), res_rmax=n("res_rmax"), res_cmax=n("res_cmax"), p=n("p"),
                            p_rmax=n("p_rmax").reshape(1, -1), p_cmax=n("p_cmax"), r=n("r"),
                            r_rmax=n("r_rmax").reshape(1, -1), r_cmax=n("r_cmax"))


def _strip_state(st, b):
    """Rows 64 b .. 64 b + 63 as a state of their own (one block row)."""
    sl = slice(64 * b, 64 * b + 64)
    return grasp.GraspState(res=st.res[sl], res_rmax=st.res_rmax[:, sl], res_cmax=st.res_cmax[b:b + 1],
                            p=st.p[sl], p_rmax=st.p_rmax[:, sl], p_cmax=st.p_cmax[b:b + 1], r=st.r, r_rmax=st.r_rmax,
                            r_cmax=st.r_cmax)


def test_grasp_llama8b_full_size():
    w = workloads.get(4)
    mats = w.matrices
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)
    rng = np.random.default_rng(32)
    grads = [workloads.make_grad(w, i, 1, device="cuda") for i in range(len(mats))]
    states = [_random_grasp_state(m.rows, m.cols, gen) for m in mats]
    host_in = {}
    picks = []
    for i, m in enumerate(mats):
        st = _grasp_host(states[i])
        for b in rng.choice((m.rows + 63) // 64, size=3, replace=False):
            sl = slice(64 * int(b), 64 * int(b) + 64)
            picks.append((i, int(b), _strip_state(st, int(b)), to_oracle_grad(grads[i][sl], "bf16").reshape(64, m.cols)))
        if i == 1:   # layer 0's k: checked whole
            host_in[i] = (st, to_oracle_grad(grads[i], "bf16").reshape(m.rows, m.cols))
    descs = [q.grasp_matrix(m.rows, m.cols, d["res"], d["res_rmax"], d["res_cmax"], d["p"], d["p_rmax"], d["p_cmax"],
                            d["r"], d["r_rmax"], d["r_cmax"], g) for m, d, g in zip(mats, states, grads)]
    ws = torch.empty(q.qmuon_grasp_workspace_size(descs), dtype=torch.uint8, device="cuda")
    q.qmuon_grasp_step(descs, 0.95, ws)
    q.qmuon_sync_status(ws)
    # M_t of sampled strips, bit-exact: it depends on the strip's state, all of
    # R and g only, so the oracle's step on the strip alone gives it
    for i, b, sst, g in picks:
        ref = grasp.grasp_step(sst, g, 0.95)
        got = grads[i][64 * b:64 * b + 64].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got, ref.m_bits, err_msg=str((i, b)))
    # one whole matrix through the oracle's step
    st, g = host_in[1]
    ref = grasp.grasp_step(st, g, 0.95)
    d = states[1]
    np.testing.assert_array_equal(grads[1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), ref.m_bits)
    gst = _grasp_host(d)
    for a_, b_ in ((gst.p, ref.state.p), (gst.r, ref.state.r), (grasp.unpack4(gst.res), grasp.unpack4(ref.state.res))):
        a_, b_ = a_.astype(np.int32), b_.astype(np.int32)
        assert np.abs(a_ - b_).max() <= 1 and np.mean(a_ == b_) >= 0.99
    np.testing.assert_allclose(gst.p_rmax, ref.state.p_rmax, rtol=1e-3)
    np.testing.assert_allclose(gst.r_rmax, ref.state.r_rmax, rtol=1e-3, atol=1e-6 * np.abs(ref.state.r_rmax).max())
