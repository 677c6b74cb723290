"""Pins for the Newton-Schulz and MuonBP oracles (CPU only).

The quintic iteration maps every singular value through the scalar
polynomial p(x) = a x + b x^3 + c x^5 and keeps the singular vectors, so the
oracle's output must equal U diag(p^k(sigma / ||G||_F)) V^T computed from a
LAPACK SVD.  That closed form, the transpose symmetry, the band that p^5
keeps normalised singular values in, and the per-iteration FLOP count of
"MuonBP ..." (section "关键设计" item 1) pin ``oracle.ns``;
``oracle.muonbp`` is pinned by the special cases P = 1 (Muon) and a 1 x 1
tiling (block step = full step), and by per-tile closed forms.
"""

import numpy as np
import pytest

from oracle import codec, muonbp, ns

A, B, C = 3.4445, -4.7750, 2.0315


def _p5(x, iters=5):
    y = np.asarray(x, dtype=np.float64)
    for _ in range(iters):
        y = A * y + B * y ** 3 + C * y ** 5
    return y


def _closed_form(G, inv=None, iters=5):
    G = np.asarray(G, np.float64)
    if inv is None:
        inv = 1.0 / (np.linalg.norm(G) + 1e-7)
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    return (U * _p5(s * inv, iters)) @ Vt


@pytest.mark.parametrize("shape", [(4, 4), (8, 16), (16, 8), (64, 96), (96, 64), (1, 7), (7, 1)])
def test_ns_equals_svd_closed_form(shape):
    rng = np.random.default_rng(sum(shape))
    G = rng.standard_normal(shape) * np.exp(rng.normal(0, 1, (shape[0], 1)))
    out = ns.newton_schulz(G)
    ref = _closed_form(G)
    assert np.linalg.norm(out - ref) <= 1e-10 * np.linalg.norm(ref)


def test_ns_explicit_inv_norm_and_iters():
    rng = np.random.default_rng(1)
    G = rng.standard_normal((12, 20))
    for iters in (1, 2, 5, 7):
        out = ns.newton_schulz(G, inv_norm=0.05, iters=iters)
        ref = _closed_form(G, inv=0.05, iters=iters)
        assert np.linalg.norm(out - ref) <= 1e-10 * np.linalg.norm(ref)


def test_ns_transpose_symmetry():
    rng = np.random.default_rng(2)
    G = rng.standard_normal((24, 40))
    np.testing.assert_allclose(ns.newton_schulz(G.T), ns.newton_schulz(G).T, rtol=0, atol=1e-12)


def test_ns_band_and_polar_factor():
    # normalised singular values in [2e-3, 1] map into [0.6818, 1.2024] after
    # five iterations (local min p(1.0501) and max p(0.5545) of the quintic)
    rng = np.random.default_rng(3)
    U, _ = np.linalg.qr(rng.standard_normal((48, 48)))
    V, _ = np.linalg.qr(rng.standard_normal((80, 48)))
    s = np.geomspace(1.0, 0.01, 48)
    G = (U * s) @ V.T
    assert s.min() / np.linalg.norm(s) >= 2e-3
    out = ns.newton_schulz(G)
    sv = np.linalg.svd(out, compute_uv=False)
    assert sv.min() >= 0.6818 and sv.max() <= 1.2024
    polar = U @ V.T
    assert np.linalg.norm(out - polar, 2) <= 0.32


def test_ns_flop_count():
    # 2(2 n m^2 + m^3) per iteration with m the smaller side
    assert ns.ns_flops(4096, 4096, 1) == 2 * (2 * 4096 ** 3 + 4096 ** 3)
    assert ns.ns_flops(14336, 4096, 1) == ns.ns_flops(4096, 14336, 1) == 2 * (2 * 14336 * 4096 ** 2 + 4096 ** 3)
    assert abs(ns.ns_flops(4096, 4096, 1) - 4.123e11) < 1e9


def _states(shapes, seed):
    rng = np.random.default_rng(seed)
    states, grads = [], []
    for r, c in shapes:
        n = r * c
        states.append(muonbp.MatrixState(r, c, np.zeros(n, np.int8),
                                         np.zeros(codec.n_blocks(n), np.float32),
                                         (rng.standard_normal((r, c)) * 0.02).astype(np.float32)))
        grads.append(codec.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32)))
    return states, grads


def test_schedule():
    assert [t for t in range(1, 21) if muonbp.is_full_step(t, 5)] == [5, 10, 15, 20]
    assert all(muonbp.is_full_step(t, 1) for t in range(1, 10))
    assert not any(muonbp.is_full_step(t, 0) for t in range(1, 50))


def test_p1_is_muon_and_1x1_tiling_is_full():
    shapes = [(32, 64), (64, 32)]
    states, grads = _states(shapes, 4)
    full, Uf, info_f = muonbp.muonbp_step(3, 1, states, grads, 0.95, 0.02, 0.005, tile=(1, 8))
    assert info_f["full"] and info_f["n_groups"] == 2
    blk, Ub, info_b = muonbp.muonbp_step(3, 0, states, grads, 0.95, 0.02, 0.02, tile=(1, 1))
    assert not info_b["full"]
    for a, b in zip(Uf, Ub):
        np.testing.assert_array_equal(a, b)
    for s0, a, b in zip(states, full, blk):
        np.testing.assert_array_equal(a.weight, b.weight)
    # the full step's update is the SVD closed form of the normalised momentum
    for k, (r, c) in enumerate(shapes):
        res = codec.momentum_update(states[k].q8, states[k].absmax, grads[k], 0.95)
        M = codec.f32_from_bf16_bits(res.grad).reshape(r, c)
        ref = _closed_form(M, inv=float(info_f["inv"][k]))
        got = codec.f32_from_bf16_bits(Uf[k]).astype(np.float64)
        assert np.linalg.norm(got - ref) <= 2 ** -8 * np.linalg.norm(ref)
        # eta_full (0.02), not eta_block, on a full step
        dW = states[k].weight.astype(np.float64) - full[k].weight
        np.testing.assert_allclose(dW, 0.02 * got, rtol=1e-6, atol=2e-8)  # one fp32 ulp of |W|


@pytest.mark.parametrize("tr,tc", [(2, 4), (4, 1)])
def test_block_step_is_per_tile_closed_form(tr, tc):
    # tile widths must be multiples of 256 (or, for row tiles, tile sizes);
    # the second matrix has tall tiles
    shapes = [(8, 1024), (600, 1024)]
    states, grads = _states(shapes, 5)
    new, U, info = muonbp.muonbp_step(2, 5, states, grads, 0.95, 0.02, 0.00707, tile=(tr, tc))
    assert not info["full"] and info["n_groups"] == 2 * tr * tc
    g = 0
    for k, (r, c) in enumerate(shapes):
        res = codec.momentum_update(states[k].q8, states[k].absmax, grads[k], 0.95)
        M = res.m.reshape(r, c).astype(np.float64)
        Mb = codec.f32_from_bf16_bits(res.grad).reshape(r, c).astype(np.float64)
        got = codec.f32_from_bf16_bits(U[k]).astype(np.float64)
        th, tw = r // tr, c // tc
        for i in range(tr):
            for j in range(tc):
                tile = M[i * th:(i + 1) * th, j * tw:(j + 1) * tw]
                inv = 1.0 / (np.linalg.norm(tile) + 1e-7)     # the tile's own norm
                assert abs(info["inv"][g] - inv) <= 1e-6 * inv
                ref = _closed_form(Mb[i * th:(i + 1) * th, j * tw:(j + 1) * tw], inv=inv)
                gt = got[i * th:(i + 1) * th, j * tw:(j + 1) * tw]
                assert np.linalg.norm(gt - ref) <= 2 ** -8 * np.linalg.norm(ref)
                g += 1
        dW = states[k].weight.astype(np.float64) - new[k].weight
        np.testing.assert_allclose(dW, 0.00707 * got, rtol=1e-6, atol=2e-8)


@pytest.mark.parametrize("rows,cols,tr,tc", [(8, 1024, 2, 4), (6, 512, 3, 1), (12, 768, 4, 3), (5, 256, 1, 1)])
def test_tile_segments_cover_exactly_their_tiles(rows, cols, tr, tc):
    # brute force: mark every element each segment names, and compare with
    # the tile (i, j) the element's row and column put it in
    segs = muonbp.tile_segments(rows, cols, tr, tc, tensor_index=3, group_base=10)
    got = np.full(rows * cols, -1)
    for s in segs:
        assert s.tensor_index == 3
        assert np.all(got[s.start:s.start + s.length] == -1)          # no element twice
        got[s.start:s.start + s.length] = s.group_id
    r, c = np.divmod(np.arange(rows * cols), cols)
    expect = 10 + (r // (rows // tr)) * tc + c // (cols // tc)
    np.testing.assert_array_equal(got, expect)
