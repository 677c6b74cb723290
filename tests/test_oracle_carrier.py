"""Pins for the MXFP8 carrier oracle (CPU only).

The E4M3 table is pinned to values fixed by the format's definition (1 sign,
4 exponent bits with bias 7, 3 mantissa bits, subnormals, 448 the largest
finite value) and the encoder to torch's own float8_e4m3fn conversion; the
scale rule and the round trip are pinned by their defining inequalities.
"""

import math

import numpy as np
import pytest
import torch

from oracle import carrier, codec

F32 = np.float32


def test_e4m3_table_fixed_points():
    t = carrier.e4m3_decode_table()
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0
    assert t[0xB8] == -1.0
    assert t[0x7E] == 448.0              # largest finite
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    finite = t[~np.isnan(t)]
    assert finite.size == 254
    assert np.all(np.diff(t[:0x7F]) > 0)  # codes 0..0x7E ascend


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, F32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_on_dense_grid():
    # every fp32 pattern whose low 12 mantissa bits are one of a few values
    # around the E4M3 rounding points, over the whole in-range binade span
    hi = np.arange(1 << 11, dtype=np.uint32) << 12
    low = np.array([0, 1, 0x7FF, 0x800, 0x801, 0xFFF], dtype=np.uint32)
    mant = (hi[:, None] | low[None, :]).reshape(-1)
    exps = np.arange(127 - 12, 127 + 9, dtype=np.uint32)  # 2^-12 .. 2^8
    bits = (exps[:, None] << 23 | mant[None, :]).reshape(-1)
    x = bits.view(F32)
    x = x[np.abs(x) <= 448.0]
    x = np.concatenate([x, -x, np.array([0.0, -0.0], F32)])
    np.testing.assert_array_equal(carrier.e4m3_encode(x), _torch_e4m3(x))


def test_e4m3_encode_is_nearest_code_by_brute_force():
    # the encoder against a search over the 127 non-negative finite codes,
    # independent of torch: the nearest value wins, a tie (exactly halfway
    # between two adjacent codes) goes to the even code, and the sign is kept
    table = carrier.e4m3_decode_table()[:0x7F].astype(np.float64)   # codes 0x00..0x7E, ascending
    rng = np.random.default_rng(11)
    mags = np.concatenate([
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)),
        (table[:-1] + table[1:]) / 2,      # every midpoint (exact in fp32)
        table,                              # every code's own value
    ]).astype(F32)
    mags = mags[mags <= 448.0]
    dist = np.abs(mags.astype(np.float64)[:, None] - table[None, :])
    nearest = dist == dist.min(axis=1, keepdims=True)
    codes = np.arange(0x7F)
    even = np.where(nearest & (codes % 2 == 0), codes, 0x7F).min(axis=1)
    pick = np.where(even == 0x7F, np.argmax(nearest, axis=1), even).astype(np.uint8)
    assert int(nearest.sum(axis=1).max()) == 2   # the midpoints really are ties
    for sign, bit in ((1.0, 0x00), (-1.0, 0x80)):
        np.testing.assert_array_equal(carrier.e4m3_encode((sign * mags).astype(F32)), pick | bit)


def test_e4m3_ties_to_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (0x38, even) and 1.125 (0x39): -> 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A, even): -> 0x3A
    assert carrier.e4m3_encode(np.array([1.0625], F32))[0] == 0x38
    assert carrier.e4m3_encode(np.array([1.1875], F32))[0] == 0x3A
    assert carrier.e4m3_encode(np.array([1000.0, -1e30], F32)).tolist() == [0x7E, 0xFE]
    assert carrier.e4m3_encode(np.array([np.nan], F32))[0] & 0x7F == 0x7F


@pytest.mark.parametrize("amax", [1e-30, 3.1e-8, 0.4375, 448.0, 449.0, 896.0, 1.0, 3.0e5, 1.7e38])
def test_block_exponent_is_minimal(amax):
    a = float(F32(amax))
    e = carrier.block_exponent(a)
    assert a <= 448.0 * 2.0 ** e
    assert a > 448.0 * 2.0 ** (e - 1)


def test_round_trip_within_half_ulp():
    rng = np.random.default_rng(0)
    rows, cols = 37, 100        # 100 = 3 full 32-blocks + a 4-wide tail per row
    m = (rng.standard_normal((rows, cols)) * np.exp(rng.normal(0, 3, (rows, 1)))).astype(F32)
    m[0, :32] = 0.0
    m[1, 5] = 1e-30
    payload, scale = carrier.encode_rows(m)
    assert payload.shape == (rows, cols) and scale.shape == (rows, 4)
    assert scale[0, 0] == 127
    vals = carrier.e4m3_decode(payload)
    assert np.all(np.abs(vals) <= 448.0)
    dec = carrier.decode_rows(payload, scale)
    # half an E4M3 ulp at the value's binade, in scaled units: ulp = 2^(E-3)
    # for normals (E = floor(log2|x|) >= -6) and 2^-9 for subnormals
    x = np.abs(m.astype(np.float64)) / carrier.e8m0_value(np.repeat(scale, 32, axis=1)[:, :cols])
    E = np.floor(np.log2(np.maximum(x, 2.0 ** -30)))
    ulp = np.where(x >= 2.0 ** -6, 2.0 ** (E - 3), 2.0 ** -9)
    err = np.abs(dec - m) / carrier.e8m0_value(np.repeat(scale, 32, axis=1)[:, :cols])
    assert np.all(err <= ulp / 2 + 1e-300)


def test_carrier_update_state_matches_codec_and_keeps_grad():
    rng = np.random.default_rng(1)
    rows, cols = 16, 96
    n = rows * cols
    g = codec.bf16_bits_from_f32(rng.standard_normal(n).astype(F32))
    q8 = np.zeros(n, np.int8)
    a = np.zeros(codec.n_blocks(n), F32)
    res = carrier.carrier_update(q8, a, g, 0.95, rows, cols)
    ref = codec.momentum_update(q8, a, g, 0.95)
    np.testing.assert_array_equal(res.q8, ref.q8)
    np.testing.assert_array_equal(res.absmax, ref.absmax)
    m64 = ref.m.astype(np.float64)
    np.testing.assert_allclose(res.inv_norm, 1 / (np.linalg.norm(m64) + 1e-7), rtol=1e-7)
    # the payload decodes to m within the E4M3 step
    dec = carrier.decode_rows(res.payload, res.scale_inv)
    rel = np.linalg.norm(dec - ref.m.reshape(rows, cols)) / np.linalg.norm(m64)
    assert rel < 2.0 ** -4
