"""MXFP8 carrier emission -- CPU oracle (test infrastructure only).

Source: "Quantized Muon Momentum", section "Wave18B MXFP8 Carrier Probe":
q8 state + grad -> q8 state + a normalised rowwise MXFP8 carrier made of an
E4M3 payload (uint8, the tensor's 2-D shape), E8M0 inverse scales (uint8,
``rows x ceil(cols / 32)``) and one fp32 inverse Frobenius norm; the gradient
buffer is not overwritten.

The page gives the container, not the encoding rules.  Readings taken:

* a scale block is 32 consecutive elements of one row; a row's last block
  may be partial and then covers only its real elements;
* the block exponent is the smallest integer ``e`` with
  ``amax <= 448 * 2**e`` (448 is the largest finite E4M3 value), so no
  element saturates; the stored E8M0 byte is ``clamp(127 + e, 0, 254)`` and
  an all-zero block stores 127;
* payload = E4M3(m / 2**(byte - 127)), rounded to nearest with ties to even
  and saturating at +-448 (NaN stays NaN, the sign of zero is kept); the
  division by a power of two is exact in fp32;
* the payload is not multiplied by the inverse norm: the normalised carrier
  is the triple (payload, scale, inv_norm);
* ``inv_norm = 1 / (sqrt(sum m*m) + 1e-7)`` over the whole tensor, with the
  same fp32 ``m`` and fp64 sum as the codec;
* the q8 state update is the codec's, unchanged.

E4M3 here is the 8-bit float with 1 sign, 4 exponent and 3 mantissa bits,
exponent bias 7, subnormals, no infinities, and only the all-ones
exponent-and-mantissa pattern reserved for NaN (so the largest finite value
is 1.75 * 2**8 = 448).  The encoder below searches the decoded code table
for the nearest value, which is the definition of round-to-nearest.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import codec

F32 = np.float32
SCALE_BLOCK = 32
E4M3_MAX = 448.0


def e4m3_decode_table() -> np.ndarray:
    """The value of every E4M3 code 0..255 (fp64; NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        mt = code & 0x7
        if e == 0xF and mt == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (mt / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + mt / 8.0) * 2.0 ** (e - 7)
    return vals


_TABLE = e4m3_decode_table()
_POS_VALUES = _TABLE[:0x7F]          # codes 0x00..0x7E: the non-negative finite values, ascending


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to E4M3 codes: nearest, ties to even, saturating.

    The magnitude is matched against the table of non-negative finite codes;
    on an exact tie between two neighbours the code with a zero last mantissa
    bit (the even code) wins.  Magnitudes above 448 saturate to 448; NaN
    encodes as 0x7F with its sign.
    """
    x = np.asarray(x, dtype=F32)
    mag = np.abs(x.astype(np.float64))
    sign = (np.signbit(x)).astype(np.uint8) << 7
    nan = np.isnan(mag)
    mag = np.where(nan, 0.0, np.minimum(mag, E4M3_MAX))
    hi = np.searchsorted(_POS_VALUES, mag, side="left")      # first value >= mag
    hi = np.clip(hi, 0, _POS_VALUES.size - 1)
    lo = np.clip(hi - 1, 0, _POS_VALUES.size - 1)
    d_hi = _POS_VALUES[hi] - mag
    d_lo = mag - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code)
    return (code | sign).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def block_exponent(amax: float) -> int:
    """Smallest integer e with amax <= 448 * 2**e (exact; amax > 0, finite)."""
    _, E = math.frexp(amax)
    e = E - 12
    while amax > math.ldexp(E4M3_MAX, e):
        e += 1
    return e


def e8m0_byte(amax: float) -> int:
    if amax == 0.0 or not math.isfinite(amax):
        return 127 if amax == 0.0 else 254
    return int(min(max(127 + block_exponent(amax), 0), 254))


def e8m0_value(byte) -> np.ndarray:
    return np.ldexp(1.0, np.asarray(byte, dtype=np.int64) - 127)


@dataclass
class CarrierResult:
    q8: np.ndarray
    absmax: np.ndarray
    m: np.ndarray            # fp32, 2-D
    payload: np.ndarray      # uint8 [rows, cols]
    scale_inv: np.ndarray    # uint8 [rows, ceil(cols/32)]
    inv_norm: np.float32
    sumsq: float


def encode_rows(m: np.ndarray):
    """Encode an fp32 matrix into (payload, scale_inv) row by row."""
    m = np.asarray(m, dtype=F32)
    rows, cols = m.shape
    nsb = (cols + SCALE_BLOCK - 1) // SCALE_BLOCK
    payload = np.zeros((rows, cols), dtype=np.uint8)
    scale = np.zeros((rows, nsb), dtype=np.uint8)
    for j in range(nsb):
        c0, c1 = j * SCALE_BLOCK, min(cols, (j + 1) * SCALE_BLOCK)
        blk = m[:, c0:c1]
        amax = np.fmax.reduce(np.abs(blk), axis=1, initial=F32(0.0))
        bytes_ = np.array([e8m0_byte(float(a)) for a in amax], dtype=np.uint8)
        scale[:, j] = bytes_
        # multiply by 2**(127 - byte): an exact power of two, representable in fp32
        mult = np.ldexp(np.float64(1.0), 127 - bytes_.astype(np.int64)).astype(F32)
        scaled = (blk * mult[:, None]).astype(F32)
        payload[:, c0:c1] = e4m3_encode(scaled)
    return payload, scale


def decode_rows(payload: np.ndarray, scale_inv: np.ndarray) -> np.ndarray:
    """payload * 2**(scale - 127), fp64."""
    rows, cols = payload.shape
    vals = e4m3_decode(payload)
    expand = np.repeat(e8m0_value(scale_inv), SCALE_BLOCK, axis=1)[:, :cols]
    return vals * expand


def carrier_update(q8: np.ndarray, absmax: np.ndarray, grad: np.ndarray, beta: float,
                   rows: int, cols: int, *, grad_dtype: str = "bf16",
                   q8_kind: str = "int8") -> CarrierResult:
    """q8 state + grad -> q8 state + (payload, scale_inv, inv_norm).

    The state update is ``codec.momentum_update`` (section "Algorithm"); the
    gradient is left as it was.
    """
    res = codec.momentum_update(q8, absmax, grad, beta, grad_dtype=grad_dtype, q8_kind=q8_kind)
    m2 = res.m.reshape(rows, cols)
    payload, scale = encode_rows(m2)
    S = float(np.sum(res.block_sumsq))
    inv = F32(1.0 / (math.sqrt(S) + codec.EPS))
    return CarrierResult(q8=res.q8, absmax=res.absmax, m=m2, payload=payload,
                         scale_inv=scale, inv_norm=inv, sumsq=S)
