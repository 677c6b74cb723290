"""Pins of the oracle's stochastic requantisation and of its generator.

The generator is pinned by the published Philox4x32-10 known-answer vectors;
the rounding by properties that fix it without restating its formula: values
already on the integer grid never move, the rounding is unbiased over many
draws and only ever picks one of the two neighbours, the clamp keeps codes in
[-127, 127], the draws depend on seed, step and tensor, and the fp64 floor
the oracle takes equals the floor in exact rational arithmetic.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codec, rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.strip() and not line.startswith("#"):
            w = [int(t, 16) for t in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,out", _kat())
def test_philox_known_answers(ctr, key, out):
    got = rng.philox4x32_10(np.array([ctr], dtype=np.uint32), key)[0]
    assert [int(x) for x in got] == out


def test_philox_rows_are_independent_of_batching():
    # a batch of counters gives each row what that counter gives alone
    ctr = np.array([[i, 7, 3, 11] for i in range(5)], dtype=np.uint32)
    whole = rng.philox4x32_10(ctr, (1, 2))
    for i in range(5):
        assert np.array_equal(rng.philox4x32_10(ctr[i:i + 1], (1, 2))[0], whole[i])


def test_uniforms_are_uniform():
    u = rng.rounding_uniforms(1 << 20, seed=12345, step=1, tensor_index=0)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))          # 24-bit grid
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / u.size)
    counts = np.bincount((u * 16).astype(int), minlength=16)
    chi2 = np.sum((counts - u.size / 16) ** 2 / (u.size / 16))
    assert chi2 < 50.0   # 15 degrees of freedom: p ~ 1e-5


def _block(values):
    """A one-block update with beta = 0 and a zero state: m equals the
    gradient, and with max|g| = 127 the requantisation factor is exactly 1."""
    g = np.zeros(256, np.float32)
    g[:len(values)] = values
    bits = codec.bf16_bits_from_f32(g)
    assert np.array_equal(codec.f32_from_bf16_bits(bits), g)   # exact in bf16
    return np.zeros(256, np.int8), np.zeros(1, np.float32), bits


def test_integers_stay_put():
    vals = [127.0, -127.0, 0.0, 5.0, -64.0, 100.0, -1.0]
    q8, a, g = _block(vals)
    for step in range(5):
        r = codec.momentum_update(q8, a, g, 0.0, rounding=codec.StochasticRounding(99, step, 3))
        assert np.array_equal(r.q8[:len(vals)].astype(np.int32), np.array(vals, dtype=np.int32))


def test_unbiased_and_only_neighbours():
    vals = [127.0, 2.25, -0.75, 10.5, -3.125, 0.0078125, -126.5]
    q8, a, g = _block(vals)
    draws = np.array([codec.momentum_update(q8, a, g, 0.0, rounding=codec.StochasticRounding(7, t, 0)).q8[:len(vals)]
                      for t in range(3000)], dtype=np.float64)
    x = np.array(vals)
    assert np.all((draws == np.floor(x)) | (draws == np.floor(x) + 1))
    frac = x - np.floor(x)
    sigma = np.sqrt(frac * (1 - frac) / draws.shape[0])
    assert np.all(np.abs(draws.mean(axis=0) - x) <= 4 * sigma + 1e-12)


def test_clamp_below_minus_127():
    # with beta = 1 the momentum is the dequantised state: code -127 (+127)
    # with block absmax A gives m = -+fl(127 * fl(A / 127)).  For an A where
    # the new absmax |m| has fl(|m| * fl(127 / |m|)) > 127, the product for
    # the element -|m| lies below -127, where floor would give -128
    A = np.random.default_rng(0).uniform(1.0, 2.0, 200000).astype(np.float32)
    s_old = (A / np.float32(127.0)).astype(np.float32)
    mabs = (np.float32(127.0) * s_old).astype(np.float32)
    sc = (np.float32(127.0) / mabs).astype(np.float32)
    hit = np.nonzero((mabs * sc).astype(np.float32) > np.float32(127.0))[0]
    assert hit.size
    a = np.array([A[hit[0]]], np.float32)
    q8 = np.zeros(256, np.int8)
    q8[0], q8[1] = -127, 127
    g = codec.bf16_bits_from_f32(np.zeros(256, np.float32))
    for step in range(50):
        r = codec.momentum_update(q8, a, g, 1.0, rounding=codec.StochasticRounding(5, step, 0))
        assert r.absmax[0] == mabs[hit[0]]
        assert int(r.q8[0]) == -127 and int(r.q8[1]) == 127


def test_draws_depend_on_seed_step_and_tensor():
    vals = [127.0] + [0.5] * 200
    q8, a, g = _block(vals)
    def codes(seed, step, t):
        return codec.momentum_update(q8, a, g, 0.0, rounding=codec.StochasticRounding(seed, step, t)).q8
    base = codes(1, 2, 3)
    assert np.array_equal(base, codes(1, 2, 3))
    for other in [codes(2, 2, 3), codes(1, 3, 3), codes(1, 2, 4), codes(1 + (1 << 32), 2, 3)]:
        assert not np.array_equal(base, other)


def test_error_below_one_step():
    rng_ = np.random.default_rng(3)
    g = codec.bf16_bits_from_f32(rng_.standard_normal(4096).astype(np.float32))
    q8 = rng_.integers(-127, 128, 4096).astype(np.int8)
    a = rng_.uniform(0.1, 2.0, 16).astype(np.float32)
    r = codec.momentum_update(q8, a, g, 0.9, rounding=codec.StochasticRounding(11, 1, 0))
    deq = codec.dequantize(r.q8, r.absmax)
    step = np.repeat(r.absmax / 127.0, 256)
    assert np.all(np.abs(r.m - deq) < step * (1 + 2 ** -20))


def test_fp64_floor_is_exact():
    # floor(x + u) of the oracle against exact rationals, on values chosen to
    # stress it: just below and above integers, tiny of both signs, and u at
    # the ends of its grid
    r = np.random.default_rng(4)
    xs = list(r.uniform(-128, 128, 3000).astype(np.float32))
    for n in range(-128, 128, 7):
        for d in (1, 2, 3):
            xs.append(np.nextafter(np.float32(n), np.float32(-1e9), dtype=np.float32) if d == 1 else
                      np.nextafter(np.float32(n), np.float32(1e9), dtype=np.float32) if d == 2 else np.float32(n))
    xs += [np.float32(v) for v in (1e-30, -1e-30, 2 ** -24, -2 ** -24, 2 ** -25, -2 ** -25, 1e-45, -1e-45)]
    us = [0, 1, 2 ** 23, 2 ** 24 - 1, 2 ** 24 - 2] + list(r.integers(0, 2 ** 24, 200))
    for i, x in enumerate(xs):
        k = int(us[i % len(us)])
        got = np.floor(np.float64(x) + k * 2.0 ** -24)
        exact = (Fraction(float(x)) + Fraction(k, 2 ** 24)).__floor__()
        assert got == exact, (x, k)


def test_exact_integer_sums_floor_to_themselves():
    # x + u landing exactly on an integer must give that integer (floor of an
    # exact sum).  With beta = 0 and fp32 gradients m = g, and with 127 in the
    # block, sc = 127/127 = 1 and x = m; x = 1 - u (exact in fp32, since u is a
    # multiple of 2^-24 below 1) then sums to exactly 1 for every element
    from oracle import rng
    seed, step, tensor = 21, 4, 2
    u = rng.rounding_uniforms(256, seed, step, tensor)
    g = (1.0 - u).astype(np.float32)
    g[0] = 127.0
    assert np.array_equal(g[1:].astype(np.float64) + u[1:], np.ones(255))
    r = codec.momentum_update(np.zeros(256, np.int8), np.zeros(1, np.float32), g, 0.0, grad_dtype="f32",
                              rounding=codec.StochasticRounding(seed, step, tensor))
    assert r.absmax[0] == 127.0
    assert int(r.q8[0]) == 127 and np.all(r.q8[1:] == 1)
