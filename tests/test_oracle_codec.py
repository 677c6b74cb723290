"""Pins for the codec oracle (CPU only).

Each test ties ``oracle.codec`` to something other than itself: the
hand-derived worked examples in ``tests/golden/``, closed forms of special
cases, error bounds of nearest rounding, torch's own bf16/fp16 rounding, and
brute-force norms.
"""

import os

import numpy as np
import pytest
import torch

from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _read_golden(name):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0][0].isalpha():
                meta[parts[0]] = [float(v) for v in parts[1:]]
            else:
                rows.append([float(v) for v in parts])
    return np.array(rows), meta


def _bf16(x):
    return codec.bf16_bits_from_f32(np.asarray(x, dtype=F32))


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_golden_beta075_ties(q8_kind):
    rows, meta = _read_golden("codec_beta075_ties.txt")
    beta = meta["beta"][0]
    idx = rows[:, 0].astype(int)
    q = np.zeros(256, dtype=np.int32)
    q[idx] = rows[:, 1]
    q8 = codec.int_to_q8(q, q8_kind)
    absmax = np.array(meta["absmax0"], dtype=F32)
    for s, (gc, mc, qc) in enumerate([(2, 3, 4), (5, 6, 7)]):
        g = np.zeros(256, dtype=F32)
        g[idx] = rows[:, gc]
        res = codec.momentum_update(q8, absmax, _bf16(g), beta, q8_kind=q8_kind)
        m_exp = np.zeros(256, dtype=F32)
        m_exp[idx] = rows[:, mc]
        q_exp = np.zeros(256, dtype=np.int32)
        q_exp[idx] = rows[:, qc]
        np.testing.assert_array_equal(res.m, m_exp)
        np.testing.assert_array_equal(codec.q8_to_int(res.q8, q8_kind), q_exp)
        np.testing.assert_array_equal(res.grad, _bf16(m_exp))
        assert res.absmax[0] == F32(meta["absmax"][s])
        assert res.block_sumsq[0] == meta["sumsq"][s]
        q8, absmax = res.q8, res.absmax


def test_golden_beta05_decay():
    rows, meta = _read_golden("codec_beta05_decay.txt")
    beta = meta["beta"][0]
    idx = rows[:, 0].astype(int)
    q = np.zeros(256, dtype=np.int32)
    q[idx] = rows[:, 1]
    q8 = codec.int_to_q8(q, "int8")
    absmax = np.array(meta["absmax0"], dtype=F32)
    g1 = np.zeros(256, dtype=F32)
    g1[idx] = rows[:, 2]
    for s in range(3):
        g = g1 if s == 0 else np.zeros(256, dtype=F32)
        res = codec.momentum_update(q8, absmax, _bf16(g), beta)
        m_exp = np.zeros(256, dtype=F32)
        m_exp[idx] = rows[:, 3 + 2 * s]
        q_exp = np.zeros(256, dtype=np.int32)
        q_exp[idx] = rows[:, 4 + 2 * s]
        np.testing.assert_array_equal(res.m, m_exp)
        np.testing.assert_array_equal(codec.q8_to_int(res.q8, "int8"), q_exp)
        assert res.absmax[0] == F32(meta["absmax"][s])
        assert res.block_sumsq[0] == meta["sumsq"][s]
        q8, absmax = res.q8, res.absmax


def test_zero_state_constant_grad():
    # old = 0 exactly, so m = fl((1 - beta) * g): one rounded product; every
    # element equal, so every code is +-127 and absmax is |m|.
    beta = F32(0.95)
    omb = F32(1.0) - beta
    assert float(omb) == 0.050000011920928955078125  # Sterbenz: 1 - 0.95f is exact
    for gval in (1e-3, -3.0, 7.5e4):
        g = np.full(256, gval, dtype=F32)
        gb = _bf16(g)
        gx = codec.f32_from_bf16_bits(gb)
        res = codec.momentum_update(np.zeros(256, np.int8), np.zeros(1, F32), gb, 0.95)
        expect = (omb * gx).astype(F32)
        np.testing.assert_array_equal(res.m, expect)
        assert res.absmax[0] == abs(expect[0])
        assert set(codec.q8_to_int(res.q8, "int8").tolist()) == {127 if gval > 0 else -127}


def test_all_zero_block_and_tail():
    # a zero block keeps absmax 0 and all-zero codes; a 17-element tail block
    # is reduced over its 17 real elements only
    rng = np.random.default_rng(0)
    n = 256 * 3 + 17
    g = np.zeros(n, dtype=F32)
    g[256:512] = rng.standard_normal(256)
    g[768:] = rng.standard_normal(17) * 10
    res = codec.momentum_update(np.zeros(n, np.int8), np.zeros(4, F32), _bf16(g), 0.9)
    assert res.absmax[0] == 0 and res.absmax[2] == 0
    assert np.all(codec.q8_to_int(res.q8, "int8")[:256] == 0)
    assert res.absmax[3] == np.max(np.abs(res.m[768:]))
    assert res.q8.size == n and res.grad.size == n
    assert np.max(np.abs(codec.q8_to_int(res.q8, "int8")[768:])) == 127


def _random_case(seed, n, q8_kind="int8"):
    rng = np.random.default_rng(seed)
    nb = codec.n_blocks(n)
    q = rng.integers(-127, 128, size=n).astype(np.int32)
    absmax = (np.abs(rng.standard_normal(nb)) * 10 ** rng.uniform(-4, 2, nb)).astype(F32)
    absmax[rng.random(nb) < 0.1] = 0
    q[np.repeat(absmax == 0, 256)[:n]] = 0
    scale = np.repeat(10 ** rng.uniform(-4, 2, nb), 256)[:n]
    g = (rng.standard_normal(n) * scale).astype(F32)
    return codec.int_to_q8(q, q8_kind), absmax, _bf16(g)


@pytest.mark.parametrize("beta", [0.95, 0.9, 0.5, 0.0, 1.0])
def test_ema_within_fp32_rounding_of_exact(beta):
    # Exact EMA of the exactly dequantised state vs the oracle's fp32 result:
    # at most one rounding of the scale, of the product, of each term and of
    # the sum -- a few ulps.  A dropped term, a sign error or beta/(1-beta)
    # swapped is off by far more.
    n = 256 * 40 + 100
    q8, absmax, gb = _random_case(1, n)
    res = codec.momentum_update(q8, absmax, gb, beta)
    q = codec.q8_to_int(q8, "int8").astype(np.float64)
    s = np.repeat(absmax.astype(np.float64) / 127.0, 256)[:n]
    old = q * s
    g = codec.f32_from_bf16_bits(gb).astype(np.float64)
    b32 = float(F32(beta))
    omb = float(F32(1.0) - F32(beta))
    exact = b32 * old + omb * g
    mag = b32 * np.abs(old) + omb * np.abs(g)
    tol = 4 * 2.0 ** -24 * mag + 1e-45
    assert np.all(np.abs(res.m.astype(np.float64) - exact) <= tol)


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_invariants(q8_kind):
    n = 256 * 64 + 33
    q8, absmax, gb = _random_case(2, n, q8_kind)
    res = codec.momentum_update(q8, absmax, gb, 0.95, q8_kind=q8_kind)
    q = codec.q8_to_int(res.q8, q8_kind)
    assert q.min() >= -127 and q.max() <= 127
    nb = codec.n_blocks(n)
    mpad = np.zeros(nb * 256, np.float64)
    mpad[:n] = res.m
    qpad = np.zeros(nb * 256, np.float64)
    qpad[:n] = q
    mb, qb = mpad.reshape(nb, 256), qpad.reshape(nb, 256)
    amax = res.absmax.astype(np.float64)
    np.testing.assert_array_equal(amax, np.max(np.abs(mb), axis=1))
    nz = amax > 0
    assert np.all(np.max(np.abs(qb[nz]), axis=1) == 127)
    assert np.all(qb[~nz] == 0)
    # nearest rounding to the grid absmax/127 * k: error at most half a step
    err = np.abs(mb - qb * (amax / 127.0)[:, None])
    assert np.all(err <= (amax / 254.0)[:, None] * (1 + 2.0 ** -20))
    # block sums are the brute-force sums of squares
    np.testing.assert_allclose(res.block_sumsq, np.sum(mb * mb, axis=1), rtol=1e-15)


def test_bf16_and_fp16_storage_match_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(1 << 16) * 10 ** rng.uniform(-30, 30, 1 << 16)).astype(F32)
    x[:4] = [0.0, -0.0, 3.4e38, -1e-45]
    # exact ties (low half 0x8000) above an even and an odd bf16, both signs
    k = (np.arange(1, 4096, dtype=np.uint32) * 7919) % 0x7F7F
    ties = ((k << 16) | 0x8000).view(F32)
    x = np.concatenate([x, ties, -ties])
    ours = codec.bf16_bits_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    y = (rng.standard_normal(1 << 14) * 100).astype(F32)
    np.testing.assert_array_equal(codec.f32_to_grad(y, "f16"),
                                  torch.from_numpy(y).half().numpy())


def test_int8_uint8_equivalent():
    n = 256 * 8 + 5
    q8, absmax, gb = _random_case(4, n, "int8")
    r_i = codec.momentum_update(q8, absmax, gb, 0.95, q8_kind="int8")
    u8 = (q8.view(np.uint8) ^ 0x80).astype(np.uint8)
    r_u = codec.momentum_update(u8, absmax, gb, 0.95, q8_kind="uint8")
    np.testing.assert_array_equal(r_i.q8.view(np.uint8) ^ 0x80, r_u.q8)
    np.testing.assert_array_equal(r_i.grad, r_u.grad)
    np.testing.assert_array_equal(r_i.absmax, r_u.absmax)


@pytest.mark.parametrize("grad_dtype", ["f16", "f32"])
def test_other_grad_dtypes_same_momentum(grad_dtype):
    # gradient values exact in bf16, f16 and f32 give the same fp32 momentum;
    # only the storage rounding of m differs
    rng = np.random.default_rng(5)
    n = 256 * 4
    q8, absmax, _ = _random_case(5, n)
    g32 = (rng.integers(-255, 256, n) * 2.0 ** rng.integers(-12, 4, n)).astype(F32)
    r_ref = codec.momentum_update(q8, absmax, _bf16(g32), 0.9)
    r = codec.momentum_update(q8, absmax, codec.f32_to_grad(g32, grad_dtype), 0.9,
                              grad_dtype=grad_dtype)
    np.testing.assert_array_equal(r.m, r_ref.m)
    np.testing.assert_array_equal(r.q8, r_ref.q8)
    np.testing.assert_array_equal(r.grad, codec.f32_to_grad(r.m, grad_dtype))


def test_group_sums_equal_bruteforce_norm():
    # interleaved QKV-like segments ("Grouped QKV And Sharding") across two tensors
    rng = np.random.default_rng(6)
    shapes = [(48, 256), (10, 100)]
    numels = [r * c for r, c in shapes]
    q8s, absmaxes, grads = [], [], []
    for k, n in enumerate(numels):
        q8, a, g = _random_case(10 + k, n)
        q8s.append(q8)
        absmaxes.append(a)
        grads.append(g)
    segs = []
    # tensor 0: rows of 256 -> blocks; split rows (2,1,1) per 4-row group like Q,K,V
    for r in range(48):
        gid = [0, 0, 1, 2][r % 4]
        segs.append(codec.NormSegment(0, r * 256, 256, gid))
    # tensor 1: one segment to the end (ends at the final partial block)
    segs.append(codec.NormSegment(1, 256, numels[1] - 256, 3))
    results, S, inv, groups = codec.multi_update(q8s, absmaxes, grads, 0.95,
                                                 segments=segs, n_groups=4)
    m0 = results[0].m.astype(np.float64).reshape(48, 256)
    for gid, rowsel in enumerate([[0, 1], [2], [3]]):
        sel = np.array([r for r in range(48) if r % 4 in rowsel])
        expect = np.linalg.norm(m0[sel]) ** 2
        np.testing.assert_allclose(S[gid], expect, rtol=1e-13)
        np.testing.assert_allclose(inv[gid], 1.0 / (np.sqrt(expect) + 1e-7), rtol=1e-7)
    m1 = results[1].m.astype(np.float64)
    np.testing.assert_allclose(S[3], np.linalg.norm(m1[256:]) ** 2, rtol=1e-13)
    # one group over everything equals the norm of the concatenation
    segs1 = [codec.NormSegment(k, 0, n, 0) for k, n in enumerate(numels)]
    _, S1, _, _ = codec.multi_update(q8s, absmaxes, grads, 0.95, segments=segs1, n_groups=1)
    allm = np.concatenate([r.m.astype(np.float64) for r in results])
    np.testing.assert_allclose(S1[0], np.dot(allm, allm), rtol=1e-13)


def test_segment_validation():
    with pytest.raises(codec.SegmentError):
        codec.block_groups([1000], [codec.NormSegment(0, 100, 200, 0)], 1)  # unaligned start
    with pytest.raises(codec.SegmentError):
        codec.block_groups([1000], [codec.NormSegment(0, 0, 300, 0)], 1)    # unaligned end
    ok = codec.block_groups([1000], [codec.NormSegment(0, 768, 232, 0)], 1)  # ends at tensor end
    assert ok[0].tolist() == [-1, -1, -1, 0]
    with pytest.raises(codec.SegmentError):
        codec.block_groups([1000], [codec.NormSegment(0, 0, 512, 0),
                                    codec.NormSegment(0, 256, 256, 1)], 2)  # overlap
    with pytest.raises(codec.SegmentError):
        codec.block_groups([1000], [codec.NormSegment(0, 0, 256, 5)], 2)    # bad group


def test_normalize_inplace():
    rng = np.random.default_rng(7)
    m = (rng.standard_normal(600) * 3).astype(F32)
    gb = _bf16(m)
    groups = np.array([0, 1, -1])
    inv = np.array([0.5, 0.25], dtype=F32)
    out = codec.normalize_inplace(gb, groups, inv)
    g32 = codec.f32_from_bf16_bits(gb)
    # scaling by a power of two is exact, so the result is the stored value scaled
    np.testing.assert_array_equal(codec.f32_from_bf16_bits(out[:256]), g32[:256] * 0.5)
    np.testing.assert_array_equal(codec.f32_from_bf16_bits(out[256:512]), g32[256:512] * 0.25)
    np.testing.assert_array_equal(out[512:], gb[512:])


def test_repeated_update_drift_is_bounded():
    # Drift of the 8-bit state away from the unquantised momentum over many
    # steps.  A requantisation moves an element by at most absmax/254 (nearest
    # rounding, 127 levels a side) and the EMA damps an earlier error by beta
    # per step, so the dequantised state never strays further than
    # max(absmax)/254/(1 - beta) from the exact fp64 EMA of the same bf16
    # gradients (fp32 rounding adds a few ulps on top).  The typical error, a
    # damped sum of independent roundings, stays near absmax/254/sqrt(3(1-beta^2)).
    rng = np.random.default_rng(5)
    n, steps, beta = 16 * 256 + 17, 100, 0.95
    nb = codec.n_blocks(n)
    scale = np.repeat(np.exp(rng.uniform(-6.0, 2.0, nb)), 256)[:n]
    bias = rng.standard_normal(n)           # a persistent direction, so the EMA settles away from 0
    q8, absmax = np.zeros(n, np.int8), np.zeros(nb, F32)
    exact = np.zeros(n)
    amax_seen = np.zeros(nb)
    rms_rel = []
    for t in range(steps):
        g = _bf16(((bias + rng.standard_normal(n)) * scale).astype(F32))
        exact = beta * exact + (1.0 - beta) * codec.f32_from_bf16_bits(g).astype(np.float64)
        r = codec.momentum_update(q8, absmax, g, beta)
        q8, absmax = r.q8, r.absmax
        amax_seen = np.maximum(amax_seen, absmax)
        drift = codec.dequantize(q8, absmax).astype(np.float64) - exact
        bound = np.repeat(amax_seen / 254.0 / (1.0 - beta), 256)[:n] * (1.0 + 1e-5) + 1e-6 * np.abs(exact)
        assert np.all(np.abs(drift) <= bound), t
        per_block = np.repeat(absmax.astype(np.float64), 256)[:n]
        rms_rel.append(np.sqrt(np.mean((drift / np.where(per_block > 0, per_block, 1.0)) ** 2)))
    typical = 1.0 / 254.0 / np.sqrt(3.0 * (1.0 - beta ** 2))
    # after a few EMA time constants it sits at the typical level and stops growing
    late, later = np.mean(rms_rel[60:80]), np.mean(rms_rel[80:])
    assert 0.7 * typical <= late <= 1.2 * typical and 0.7 * typical <= later <= 1.2 * typical
    assert abs(later - late) <= 0.1 * late


def test_inverse_norm_adds_eps_to_the_norm():
    # the reading inv = 1/(||m|| + 1e-7), epsilon added to the norm: an empty
    # (all-zero) group gives 1e7 exactly, and a group of 256 values 2^-10
    # (sum of squares 2^-12, norm 2^-6) gives 1/(2^-6 + 1e-7) = 64/(1 + 6.4e-6)
    # = 63.99959040262142...; epsilon under the root would give 3162.3 and 63.987
    q8, a = np.zeros(512, np.int8), np.zeros(2, F32)
    g = np.zeros(512, F32)
    g[256:] = 2.0 ** -10
    r = codec.momentum_update(q8, a, _bf16(g), 0.0)          # beta = 0: m = g exactly
    groups = codec.block_groups([512], [codec.NormSegment(0, 0, 256, 0), codec.NormSegment(0, 256, 256, 1)], 2)
    S, inv = codec.group_sumsq([r.block_sumsq], groups, 2)
    assert S.tolist() == [0.0, 2.0 ** -12]
    assert inv[0] == F32(1e7)
    assert inv[1] == F32(63.99959040262142)


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_dequantize_fixed_points(q8_kind):
    # step 2's scale is absmax/127: with absmax 127 every code dequantises to
    # itself, with absmax 254 to twice itself (both exact in fp32), with absmax
    # 0 to zero, and the ends +-127 always give +-absmax
    q = np.arange(-127, 128, dtype=np.int32)
    q = np.concatenate([q, q[:1]])                          # 256 codes = one block
    codes = codec.int_to_q8(q, q8_kind)
    for amax, mult in ((127.0, 1.0), (254.0, 2.0), (0.0, 0.0)):
        d = codec.dequantize(codes, np.array([amax], F32), q8_kind)
        assert np.array_equal(d, (q * mult).astype(F32)), amax
    for amax in (0.37, 1e-20, 3e30):
        d = codec.dequantize(codes, np.array([amax], F32), q8_kind)
        assert abs(d[0] + F32(amax)) <= F32(amax) * 2 ** -23     # code -127: two roundings of -absmax
        assert abs(d[254] - F32(amax)) <= F32(amax) * 2 ** -23


def test_nonfinite_momentum_readings():
    # the readings for non-finite momenta: the absmax ignores NaN lanes (an
    # all-NaN block gets 0), a NaN product gives code 0, and an infinity makes
    # the absmax infinite and every code of its block 0.  beta = 0, so m = g
    g = np.zeros(768, F32)
    g[0], g[1], g[2] = np.nan, 2.0, -1.0          # block 0: NaN among finite values
    g[256:512] = np.nan                           # block 1: NaN only
    g[512], g[513] = np.inf, 3.0                  # block 2: an infinity
    r = codec.momentum_update(np.zeros(768, np.int8), np.zeros(3, F32), g, 0.0, grad_dtype="f32")
    assert r.absmax.tolist() == [2.0, 0.0, np.inf]
    q = r.q8.astype(np.int32)
    assert q[0] == 0 and q[1] == 127 and q[2] == -64          # -1 * 63.5 = -63.5 -> -64 (ties to even)
    assert np.all(q[256:512] == 0) and np.all(q[512:] == 0)
    assert np.isnan(r.block_sumsq[0]) and np.isnan(r.block_sumsq[1]) and r.block_sumsq[2] == np.inf
