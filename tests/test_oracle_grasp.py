"""Pins of the GRASP oracle (4-bit residual + rank-k factor, grid quantisation).

Grid quantisation is pinned by its definition checked element by element on a
brute-force loop, exactness on its own grid, the half-step error bound, and
the property it is there for (an outlier row and column leave the rest of the
block finely resolved, unlike one scale per block); the power iteration by
orthonormality, the residual being orthogonal to span(P), and convergence of
the captured energy to the top-k singular values of an SVD; the momentum
step by its zero-state and mu = 0 special cases and by a rank-k gradient whose
residual vanishes.
"""

import numpy as np
import pytest

from oracle import codec, grasp


def test_grid_quantize_matches_brute_force():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((70, 90)) * np.exp(rng.uniform(-3, 3, (70, 1)))).astype(np.float32)
    s_r, s_c, bits = 32, 16, 4
    q, rmax, cmax = grasp.grid_quantize(x, bits, s_r, s_c)
    L = np.float32(7)
    for i in range(70):
        for j in range(90):
            bi, bj = i // s_r, j // s_c
            blk = np.abs(x[bi * s_r:(bi + 1) * s_r, bj * s_c:(bj + 1) * s_c])
            r = blk[i - bi * s_r, :].max()
            c = blk[:, j - bj * s_c].max()
            d = min(r, c)
            assert rmax[bj, i] == r and cmax[bi, j] == c
            want = 0 if d == 0 else int(np.clip(np.rint(np.float32(x[i, j] * np.float32(L / np.float32(d)))), -7, 7))
            assert q[i, j] == want


def test_grid_exact_on_its_grid_and_zero_blocks():
    a = np.float32(0.75)
    x = np.where(np.random.default_rng(1).random((64, 64)) < 0.5, a, -a).astype(np.float32)
    x[:, 40:] = 0.0   # a zero column block inside the first row block
    q, rmax, cmax = grasp.grid_quantize(x, 8, 64, 32)
    back = grasp.grid_dequantize(q, rmax, cmax, 8, 64, 32)
    assert np.array_equal(back, x)
    assert np.all(q[:, 40:] == 0)


def test_grid_error_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((300, 260)).astype(np.float32)
    x[rng.random(x.shape) < 0.001] *= 1000.0   # outliers
    for bits in (4, 8):
        L = 2 ** (bits - 1) - 1
        q, rmax, cmax = grasp.grid_quantize(x, bits, 64, 64)
        back = grasp.grid_dequantize(q, rmax, cmax, bits, 64, 64)
        d = grasp._block_min(rmax, cmax, 300, 260, 64, 64)
        assert np.all(np.abs(back - x) <= 0.5 * d / L * (1 + 2 ** -20))


@pytest.mark.parametrize("axis", [0, 1])
def test_grid_confines_outliers(axis):
    # an outlier row (or column) in a block: one scale per block would round
    # everything else to zero; with the smaller of row and column maxima the
    # rest of the block keeps its resolution
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, (64, 64)).astype(np.float32)
    if axis == 0:
        x[5, :] *= 1e4
    else:
        x[:, 9] *= 1e4
    q, rmax, cmax = grasp.grid_quantize(x, 4, 64, 64)
    back = grasp.grid_dequantize(q, rmax, cmax, 4, 64, 64)
    rest = np.ones_like(x, bool)
    if axis == 0:
        rest[5, :] = False
    else:
        rest[:, 9] = False
    err_grid = np.abs(back - x)[rest].max()
    amax = np.abs(x).max()
    err_block = np.abs(np.rint(x / amax * 7) * amax / 7 - x)[rest].max()
    assert err_grid <= 0.5 / 7 * 1.0001 and err_block > 0.9


def test_pack4_round_trip():
    q = np.tile(np.arange(-7, 8, dtype=np.int8), (3, 2))[:, :30]
    assert np.array_equal(grasp.unpack4(grasp.pack4(q)), q)
    assert grasp.pack4(np.array([[-7, 7]], np.int8))[0, 0] == (1 | (15 << 4))


def test_orthonormal_factor():
    rng = np.random.default_rng(4)
    y = rng.standard_normal((200, 8))
    p = grasp.orthonormal_factor(y)
    assert np.allclose(p.T @ p, np.eye(8), atol=1e-12)
    assert np.allclose(p @ (p.T @ y), y, atol=1e-10)        # same column space
    assert np.all(np.diag(p.T @ y) > 0)                     # positive triangular diagonal


def _state(rows, cols, seed, k=8):
    return grasp.initial_state(rows, cols, np.random.default_rng(seed).standard_normal((cols, k)).astype(np.float32), k)


def test_first_step_and_mu_zero():
    rng = np.random.default_rng(5)
    rows, cols = 96, 140
    g = codec.bf16_bits_from_f32(rng.standard_normal(rows * cols).astype(np.float32))
    out = grasp.grasp_step(_state(rows, cols, 6), g, 0.9)
    assert np.array_equal(out.m_bits.reshape(-1), g)          # zero state: M_1 = g
    g2 = codec.bf16_bits_from_f32(rng.standard_normal(rows * cols).astype(np.float32))
    out2 = grasp.grasp_step(out.state, g2, 0.0)
    assert np.array_equal(out2.m_bits.reshape(-1), g2)        # mu = 0 ignores the state


def test_residual_orthogonal_to_p():
    rng = np.random.default_rng(7)
    rows, cols = 150, 100
    g = codec.bf16_bits_from_f32(rng.standard_normal(rows * cols).astype(np.float32))
    out = grasp.grasp_step(_state(rows, cols, 8), g, 0.9)
    scale = np.linalg.norm(out.res)
    assert np.abs(out.p.T @ out.res).max() < 1e-10 * scale


def test_power_iteration_converges_to_top_k():
    # fixed M with a spectral gap: repeated warm-started steps capture the
    # top-k singular energy (here without quantisation, the linear algebra alone)
    rng = np.random.default_rng(9)
    rows, cols, k = 120, 90, 8
    u, _ = np.linalg.qr(rng.standard_normal((rows, rows)))
    v, _ = np.linalg.qr(rng.standard_normal((cols, cols)))
    sig = np.concatenate([np.linspace(10, 6, k), np.linspace(1, 0.1, cols - k)])
    m = (u[:, :cols] * sig) @ v.T
    r = rng.standard_normal((cols, k))
    energy = []
    for _ in range(12):
        q = r / np.linalg.norm(r, axis=0)
        p = grasp.orthonormal_factor(m @ q)
        r = m.T @ p
        energy.append(np.linalg.norm(p @ r.T) ** 2)
    top = np.sum(sig[:k] ** 2)
    assert all(b >= a - 1e-9 for a, b in zip(energy, energy[1:]))
    assert abs(energy[-1] - top) < 1e-6 * top


def test_low_rank_gradient_leaves_small_residual():
    rng = np.random.default_rng(10)
    rows, cols, k = 128, 192, 8
    a = rng.standard_normal((rows, k)).astype(np.float32)
    b = rng.standard_normal((cols, k)).astype(np.float32)
    g = codec.bf16_bits_from_f32((a @ b.T).astype(np.float32).reshape(-1))
    st = _state(rows, cols, 11, k)
    for _ in range(3):
        out = grasp.grasp_step(st, g, 0.9)
        st = out.state
    mt = codec.f32_from_bf16_bits(out.m_bits).astype(np.float64)
    assert np.linalg.norm(out.res) < 0.01 * np.linalg.norm(mt)


def test_state_reconstructs_the_momentum():
    # the stored state (grid-quantised 4-bit residual and 8-bit factors)
    # dequantises to M_t up to quantisation error, which is small next to the
    # rank-k part it carries; here a rank-8 signal plus noise over three steps
    # with mu = 0.9, so the reconstruction of M_{t-1} feeds every later step
    rng = np.random.default_rng(12)
    rows, cols, k = 160, 128, 8
    low = rng.standard_normal((rows, k)) @ rng.standard_normal((k, cols))
    st = _state(rows, cols, 13, k)
    for _ in range(3):
        g = codec.bf16_bits_from_f32((low + 0.3 * rng.standard_normal((rows, cols))).astype(np.float32).reshape(-1))
        out = grasp.grasp_step(st, g, 0.9)
        st = out.state
    mt = codec.f32_from_bf16_bits(out.m_bits).astype(np.float64)
    rec = grasp.reconstruct(*grasp.dequantize_parts(st)).astype(np.float64)
    assert np.linalg.norm(rec - mt) < 0.02 * np.linalg.norm(mt)          # measured 0.8%
    assert np.linalg.norm(out.p @ out.r.T) > 0.9 * np.linalg.norm(mt)   # the factor carries the signal
