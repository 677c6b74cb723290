"""GPU parity of the GRASP momentum step (qmuon_grasp_step) against the oracle.

M_t, stored in bf16 over the gradient, is bit-exact: the reconstruction and
the momentum follow the oracle's operations and order.  The power iteration
and the residual come from different floating-point paths (fp32 tiles and a
CholeskyQR2 here, an fp64 QR in the oracle).  A code is rint(t) with
t = x * fl(L / d); the GPU's t differs from the oracle's by the propagated
fp32 rounding, |dt| <= L (|dx| + |x| |dd| / d) / d, which is at most
2 L rho max / d when rho bounds the relative perturbation of the block's
values (measured here on the stored maxima).  So the new codes are held to:
none off by more than one level, every differing code a near tie of the
oracle's t (within that band of a half-integer, with a safety factor), at
least 99% identical, and a reconstruction of M_t as close as the oracle's own.
"""

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
from oracle import codec, grasp

pytestmark = pytest.mark.gpu

# ragged strips (200, 1000 and 201 rows; 201 and 9 also leave half a row pair
# empty), a single block, one row more than the factor's rank (with exactly 8
# rows the residual is zero up to rounding and its codes quantise noise), and
# a tall matrix whose last 128-row chunk of R's sums holds 4 rows
SHAPES = [(128, 192), (200, 320), (64, 64), (1000, 128), (1024, 2048), (201, 192), (9, 64), (4100, 128)]


def _to_dev(st, grad_bits, rows, cols):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d = dict(res=t(st.res), res_rmax=t(st.res_rmax), res_cmax=t(st.res_cmax), p=t(st.p), p_rmax=t(st.p_rmax),
             p_cmax=t(st.p_cmax), r=t(st.r), r_rmax=t(st.r_rmax), r_cmax=t(st.r_cmax),
             grad=torch.from_numpy(grad_bits.astype(np.int16).reshape(rows, cols)).cuda().view(torch.bfloat16))
    return d


def _desc(d, rows, cols):
    return q.grasp_matrix(rows, cols, d["res"], d["res_rmax"], d["res_cmax"], d["p"], d["p_rmax"], d["p_cmax"],
                          d["r"], d["r_rmax"], d["r_cmax"], d["grad"])


def _from_dev(d):
    n = lambda k: d[k].cpu().numpy()
    return grasp.GraspState(res=n("res"), res_rmax=n("res_rmax"), res_cmax=n("res_cmax"), p=n("p"),
                            p_rmax=n("p_rmax"), p_cmax=n("p_cmax"), r=n("r"), r_rmax=n("r_rmax"),
                            r_cmax=n("r_cmax"))


def _grad(rows, cols, seed):
    r = np.random.default_rng(seed)
    x = r.standard_normal((rows, cols)).astype(np.float32)
    x += 3.0 * np.outer(r.standard_normal(rows), r.standard_normal(cols)).astype(np.float32)   # a dominant direction
    return codec.bf16_bits_from_f32(x.reshape(-1)).reshape(rows, cols)


def _codes_close(a, b):
    a, b = a.astype(np.int32), b.astype(np.int32)
    assert np.abs(a - b).max() <= 1
    assert np.mean(a == b) >= 0.99


def _rel(got, want):
    """Largest relative difference of stored maxima (where the oracle's are nonzero)."""
    w = np.abs(want.astype(np.float64))
    keep = w > 0
    return float(np.max(np.abs(got.astype(np.float64)[keep] - w[keep]) / w[keep])) if keep.any() else 0.0


def _ties_explain_flips(x, rmax, cmax, bits, s_rows, s_cols, got_codes, rho, safety=8.0):
    """Every code where the GPU differs from the oracle is a near tie: the
    oracle's t = x * fl(L / d) lies within safety * 2 L rho (max/d) (+ two fp32
    roundings of t) of a half-integer, max being the larger of the element's
    row and column maxima in its block."""
    x = np.asarray(x, np.float32)
    R, C = x.shape
    L = np.float32(2 ** (bits - 1) - 1)
    rb = np.repeat(rmax.T, s_cols, axis=1)[:, :C]
    cb = np.repeat(cmax, s_rows, axis=0)[:R, :]
    d = np.minimum(rb, cb).astype(np.float32)
    big = np.maximum(rb, cb).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (x * np.where(d == 0, np.float32(0), (L / np.where(d == 0, np.float32(1), d)).astype(np.float32))
             ).astype(np.float64)
        ref = np.clip(np.rint(t), -L, L)
        band = safety * 2.0 * float(L) * rho * np.where(d > 0, big / d, 0.0) + float(L) * 2.0 ** -21
    diff = got_codes.astype(np.int32) != ref.astype(np.int32)
    if diff.any():
        dist = np.abs(np.abs(t - np.floor(t)) - 0.5)
        worst = float(np.max(dist[diff] - band[diff]))
        assert worst <= 0.0, (int(diff.sum()), worst)


def _run_step(states, grads, mu):
    devs = [_to_dev(st, g, *g.shape) for st, g in zip(states, grads)]
    descs = [_desc(d, *g.shape) for d, g in zip(devs, grads)]
    ws = torch.empty(q.qmuon_grasp_workspace_size(descs), dtype=torch.uint8, device="cuda")
    q.qmuon_grasp_step(descs, mu, ws)
    q.qmuon_sync_status(ws)
    return devs


@pytest.mark.parametrize("warm", [False, True])
def test_grasp_step_matches_oracle(warm):
    states, grads = [], []
    for i, (rows, cols) in enumerate(SHAPES):
        st = grasp.initial_state(rows, cols, np.random.default_rng(50 + i).standard_normal((cols, 8)).astype(np.float32))
        if warm:   # a state with a non-zero residual and factor: one oracle step first
            st = grasp.grasp_step(st, _grad(rows, cols, 70 + i), 0.9).state
        states.append(st)
        grads.append(_grad(rows, cols, 90 + i))
    devs = _run_step(states, grads, 0.9)
    for (rows, cols), st, g, d in zip(SHAPES, states, grads, devs):
        ref = grasp.grasp_step(st, g, 0.9)
        got_m = d["grad"].view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got_m, ref.m_bits)
        gst = _from_dev(d)
        _codes_close(gst.p, ref.state.p)
        _codes_close(gst.r, ref.state.r)
        _codes_close(grasp.unpack4(gst.res), grasp.unpack4(ref.state.res))
        rho_p = max(_rel(gst.p_rmax, ref.state.p_rmax), _rel(gst.p_cmax, ref.state.p_cmax))
        rho_r = max(_rel(gst.r_rmax, ref.state.r_rmax), _rel(gst.r_cmax, ref.state.r_cmax))
        rho_res = max(_rel(gst.res_rmax, ref.state.res_rmax), _rel(gst.res_cmax, ref.state.res_cmax), rho_p, rho_r)
        _ties_explain_flips(ref.p, ref.state.p_rmax, ref.state.p_cmax, 8, 64, 8, gst.p, rho_p)
        _ties_explain_flips(ref.r, ref.state.r_rmax, ref.state.r_cmax, 8, 64, 8, gst.r, rho_r)
        if rows > 8:   # with exactly 8 rows the residual is rounding noise
            _ties_explain_flips(ref.res, ref.state.res_rmax, ref.state.res_cmax, 4, 64, 64, grasp.unpack4(gst.res),
                                rho_res)
        # the factors' maxima: Y = M_t Q is fp32 here and fp64 in the oracle, and
        # the orthogonalisation scales its relative error by the condition
        # number of M_t Q (large when one direction dominates, as here): 1e-3,
        # an eighth of one 8-bit level
        np.testing.assert_allclose(gst.p_rmax, ref.state.p_rmax, rtol=1e-3)
        np.testing.assert_allclose(gst.r_rmax, ref.state.r_rmax, rtol=1e-3, atol=1e-6 * np.abs(ref.state.r_rmax).max())
        # the stored state reconstructs M_t as well as the oracle's does
        mt = codec.f32_from_bf16_bits(ref.m_bits).astype(np.float64)
        def err(s):
            res, p, r = grasp.dequantize_parts(s)
            return np.linalg.norm(res.astype(np.float64) + p.astype(np.float64) @ r.astype(np.float64).T - mt)
        assert err(gst) <= 1.05 * err(ref.state) + 1e-9 * np.linalg.norm(mt)


def test_grasp_three_steps_track_the_oracle():
    rows, cols = 512, 768
    st_host = grasp.initial_state(rows, cols, np.random.default_rng(1).standard_normal((cols, 8)).astype(np.float32))
    st_dev = st_host
    for t in range(3):
        g = _grad(rows, cols, 200 + t)
        d = _run_step([st_dev], [g], 0.95)[0]
        st_dev = _from_dev(d)
        ref = grasp.grasp_step(st_host, g, 0.95)
        st_host = ref.state
        got = codec.f32_from_bf16_bits(d["grad"].view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
        want = codec.f32_from_bf16_bits(ref.m_bits).astype(np.float64)
        assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want), t


def test_grasp_rejects_bad_shapes():
    rows, cols = 64, 100   # cols not a multiple of 64
    st = grasp.initial_state(rows, cols, np.ones((cols, 8), np.float32))
    d = _to_dev(st, np.zeros((rows, cols), np.uint16), rows, cols)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_grasp_step([_desc(d, rows, cols)], 0.9, ws)
    assert e.value.status == q.QMUON_ERR_UNSUPPORTED
    rows, cols = 7, 64     # fewer rows than the factor's rank
    st = grasp.initial_state(rows, cols, np.ones((cols, 8), np.float32))
    d = _to_dev(st, np.zeros((rows, cols), np.uint16), rows, cols)
    with pytest.raises(q.QmuonError) as e:
        q.qmuon_grasp_step([_desc(d, rows, cols)], 0.9, ws)
    assert e.value.status == q.QMUON_ERR_INVALID_ARGUMENT


def test_grasp_step_does_not_depend_on_workspace_contents():
    # the same warm step with every workspace byte zeroed and then set to 0xFF
    # (NaN in every float scratch) leaves bit-identical states and M_t: each
    # scratch value (strip shares, Gram sums, factors) is written before it is read
    shapes = [(200, 320), (1000, 128), (1024, 2048), (9, 64)]
    states, grads = [], []
    for i, (rows, cols) in enumerate(shapes):
        st = grasp.initial_state(rows, cols, np.random.default_rng(60 + i).standard_normal((cols, 8)).astype(np.float32))
        states.append(grasp.grasp_step(st, _grad(rows, cols, 80 + i), 0.9).state)
        grads.append(_grad(rows, cols, 100 + i))
    outs = []
    for fill in (0x00, 0xFF):
        devs = [_to_dev(st, g, *g.shape) for st, g in zip(states, grads)]
        descs = [_desc(d, *g.shape) for d, g in zip(devs, grads)]
        ws = torch.full((q.qmuon_grasp_workspace_size(descs),), fill, dtype=torch.uint8, device="cuda")
        q.qmuon_grasp_step(descs, 0.9, ws)
        q.qmuon_sync_status(ws)
        outs.append(devs)
    for da, db in zip(*outs):
        for k in da:
            assert torch.equal(da[k].contiguous().view(torch.uint8), db[k].contiguous().view(torch.uint8)), k
