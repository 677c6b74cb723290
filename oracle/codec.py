"""Blockwise 8-bit Muon momentum codec -- CPU oracle (test infrastructure only).

Source: "Quantized Muon Momentum" (cppmega docs), section "Algorithm",
steps 1-9, and the state format listed under "What Exists" (int8/uint8
payload of the momentum's shape, one fp32 absmax per 256 elements,
symmetric nearest rounding to [-127, 127]).  Grouped sums follow section
"Grouped QKV And Sharding" (norm segments, one group id per 256-element
block, segment boundaries on block boundaries except at a tensor's final
partial block).

All codec arithmetic is IEEE fp32 with one rounding per operation, in the
order written below; numpy performs each ufunc separately, so nothing is
contracted into a fused multiply-add.  Readings taken where the page is
silent:

* dequantisation: ``s = absmax / 127`` (one correctly rounded division per
  block), then ``old = float(q) * s``;
* ``omb = 1 - beta`` in fp32, then ``m = (beta * old) + (omb * g)`` -- the
  exponential-moving-average form of step 4, not a ``lerp``;
* new absmax = max |m| over the fp32 values (maxNum semantics: a NaN lane is
  ignored, an all-NaN block gives 0);
* requantisation: ``sc = 127 / amax`` (one division per block), then
  ``q = clamp(rint(m * sc), -127, 127)`` with ties to even; a NaN product
  gives 0; ``amax == 0`` gives all-zero codes;
* uint8 storage is offset binary, ``u = q + 128`` (int8 bits XOR 0x80);
* the per-block sum of squares is taken over the fp32 ``m`` (step 9) and
  accumulated in fp64; a group's inverse norm is ``1 / (sqrt(S) + 1e-7)``
  evaluated in fp64 and rounded once to fp32.

Stochastic requantisation (optional; the page's section "Known Limitations" says
only that it is not implemented yet): with ``x = m * sc`` as above and a
uniform ``u`` in [0, 1) per element (``oracle.rng``: Philox4x32-10 keyed by
the seed, counter from the element, tensor and step), ``q = clamp(floor(x +
u), -127, 127)``, a NaN product giving 0.  ``x + u`` is evaluated in fp64,
where it is exact enough for the floor: the exact sum lies on the grid of
min(ulp(x), 2^-24) and never falls within fp64's rounding error of an
integer it does not reach.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import rng

QBLOCK = 256
EPS = 1e-7
F32 = np.float32

GRAD_DTYPES = ("bf16", "f16", "f32")
Q8_KINDS = ("int8", "uint8")


# --------------------------------------------------------------------------
# bf16 / fp16 storage helpers (bf16 is carried as its uint16 bit pattern)
# --------------------------------------------------------------------------

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest, ties to even); returns uint16 bits.

    bfloat16 is the top half of an IEEE binary32, so rounding keeps the high
    16 bits after adding half an ulp of the low half (plus the tie-to-even
    bias).  NaN maps to a quiet NaN with the input's sign.
    """
    x = np.ascontiguousarray(x, dtype=F32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        sign = ((u >> 16) & 0x8000).astype(np.uint16)
        rounded = np.where(nan, sign | np.uint16(0x7FC0), rounded)
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(F32)


def grad_to_f32(grad: np.ndarray, grad_dtype: str) -> np.ndarray:
    """Widen a gradient buffer to fp32 (exact for every supported dtype)."""
    if grad_dtype == "bf16":
        return f32_from_bf16_bits(grad)
    if grad_dtype == "f16":
        return np.asarray(grad, dtype=np.float16).astype(F32)
    if grad_dtype == "f32":
        return np.asarray(grad, dtype=F32).copy()
    raise ValueError(f"unknown grad dtype {grad_dtype!r}")


def f32_to_grad(m: np.ndarray, grad_dtype: str) -> np.ndarray:
    """Store fp32 values in the gradient dtype (step 5 of "Algorithm")."""
    if grad_dtype == "bf16":
        return bf16_bits_from_f32(m)
    if grad_dtype == "f16":
        return np.asarray(m, dtype=F32).astype(np.float16)  # IEEE nearest-even
    if grad_dtype == "f32":
        return np.asarray(m, dtype=F32).copy()
    raise ValueError(f"unknown grad dtype {grad_dtype!r}")


def q8_to_int(q8: np.ndarray, q8_kind: str) -> np.ndarray:
    """Decode stored codes to signed integers in [-127, 127]."""
    if q8_kind == "int8":
        return np.asarray(q8, dtype=np.int8).astype(np.int32)
    if q8_kind == "uint8":
        return np.asarray(q8, dtype=np.uint8).astype(np.int32) - 128
    raise ValueError(f"unknown q8 kind {q8_kind!r}")


def int_to_q8(q: np.ndarray, q8_kind: str) -> np.ndarray:
    """Encode signed integers in [-127, 127] into the stored code type."""
    q = np.asarray(q, dtype=np.int32)
    if q8_kind == "int8":
        return q.astype(np.int8)
    if q8_kind == "uint8":
        return (q + 128).astype(np.uint8)
    raise ValueError(f"unknown q8 kind {q8_kind!r}")


def n_blocks(numel: int) -> int:
    return (int(numel) + QBLOCK - 1) // QBLOCK


# --------------------------------------------------------------------------
# The per-block update ("Algorithm", steps 1-9)
# --------------------------------------------------------------------------

@dataclass
class UpdateResult:
    q8: np.ndarray          # new codes, same dtype/shape as the input codes (flat)
    absmax: np.ndarray      # fp32 [nb]
    m: np.ndarray           # fp32 momentum (flat), before storage rounding
    grad: np.ndarray        # m stored in the gradient dtype (flat)
    block_sumsq: np.ndarray  # fp64 [nb], sum of m*m per block


def _pad_blocks(x: np.ndarray, numel: int, fill=0) -> np.ndarray:
    nb = n_blocks(numel)
    out = np.full(nb * QBLOCK, fill, dtype=x.dtype)
    out[:numel] = x.reshape(-1)[:numel]
    return out.reshape(nb, QBLOCK)


def dequantize(q8: np.ndarray, absmax: np.ndarray, q8_kind: str = "int8") -> np.ndarray:
    """Steps 1-2: old = float(q) * (absmax / 127), fp32, per 256-block."""
    q8 = np.asarray(q8).reshape(-1)
    numel = q8.size
    qv = _pad_blocks(q8_to_int(q8, q8_kind), numel).astype(F32)
    s_old = (np.asarray(absmax, dtype=F32) / F32(127.0)).astype(F32)
    old = qv * s_old[:, None]
    return old.reshape(-1)[:numel]


@dataclass(frozen=True)
class StochasticRounding:
    """Stochastic requantisation of one tensor: the generator's key and the
    step and tensor words of its counter."""
    seed: int
    step: int
    tensor_index: int = 0


def momentum_update(q8: np.ndarray, absmax: np.ndarray, grad: np.ndarray, beta: float,
                    *, grad_dtype: str = "bf16", q8_kind: str = "int8",
                    rounding: Optional[StochasticRounding] = None) -> UpdateResult:
    """One quantized momentum update of a flat tensor.

    Follows "Quantized Muon Momentum", section "Algorithm": load the codes and
    the block absmax (1), dequantise in fp32 (2), load the gradient (3),
    ``m = beta * old_m + (1 - beta) * grad`` (4), store ``m`` over the
    gradient (5), take the new block absmax (6), requantise (7), store codes
    and absmax (8), and the block sum of squares (9).  The last block of a
    tensor whose size is not a multiple of 256 holds only its real elements.
    With ``rounding`` set, step 7 rounds stochastically (module docstring).
    """
    q8 = np.asarray(q8).reshape(-1)
    numel = q8.size
    nb = n_blocks(numel)
    absmax = np.asarray(absmax, dtype=F32).reshape(-1)
    if absmax.size != nb:
        raise ValueError(f"absmax has {absmax.size} entries, expected {nb}")
    g32 = grad_to_f32(np.asarray(grad).reshape(-1), grad_dtype)
    if g32.size != numel:
        raise ValueError("grad and q8 sizes differ")

    # (1)-(2) dequantise: one division per block, one multiply per element
    qv = _pad_blocks(q8_to_int(q8, q8_kind), numel).astype(F32)
    s_old = (absmax / F32(127.0)).astype(F32)
    old = (qv * s_old[:, None]).astype(F32)

    # (3)-(4) EMA in fp32: two rounded products, one rounded sum
    beta32 = F32(beta)
    omb = F32(F32(1.0) - beta32)
    g = _pad_blocks(g32, numel)
    m = ((beta32 * old).astype(F32) + (omb * g).astype(F32)).astype(F32)
    if numel % QBLOCK:
        m.reshape(-1)[numel:] = 0.0  # padding lanes are not part of the tensor

    # (6) new absmax over fp32 m, NaN lanes ignored
    amax = np.fmax.reduce(np.abs(m), axis=1, initial=F32(0.0)).astype(F32)

    # (7) requantise: sc = 127 / amax per block, q = clamp(rint(m * sc))
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        sc = np.where(amax == 0, F32(0.0), F32(127.0) / np.where(amax == 0, F32(1.0), amax)).astype(F32)
        x = (m * sc[:, None]).astype(F32)
        if rounding is None:
            r = np.rint(x)
        else:
            u = _pad_blocks(rng.rounding_uniforms(numel, rounding.seed, rounding.step, rounding.tensor_index),
                            numel)
            r = np.floor(x.astype(np.float64) + u)
        r = np.where(np.isnan(r), 0.0, r)
        qn = np.clip(r, -127, 127).astype(np.int32)
    qn = np.where(amax[:, None] == 0, 0, qn)

    # (9) block sum of squares of the fp32 momentum, fp64 accumulation
    m64 = m.astype(np.float64)
    block_sumsq = np.sum(m64 * m64, axis=1)

    m_flat = m.reshape(-1)[:numel].copy()
    return UpdateResult(
        q8=int_to_q8(qn.reshape(-1)[:numel], q8_kind),
        absmax=amax,
        m=m_flat,
        grad=f32_to_grad(m_flat, grad_dtype),          # (5)
        block_sumsq=block_sumsq,
    )


# --------------------------------------------------------------------------
# Norm groups ("Grouped QKV And Sharding")
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class NormSegment:
    """A run of one tensor's flat elements that belongs to a norm group."""
    tensor_index: int
    start: int
    length: int
    group_id: int


class SegmentError(ValueError):
    pass


def block_groups(numels: Sequence[int], segments: Optional[Sequence[NormSegment]],
                 n_groups: int) -> list:
    """Map every 256-element block of every tensor to its norm group.

    ``segments=None`` puts each tensor in its own group (group id = tensor
    index).  Otherwise each segment must start on a block boundary and end on
    one, or at the end of its tensor; blocks covered by no segment belong to
    no group (-1).  A block covered twice is an error.
    """
    out = [np.full(n_blocks(n), -1, dtype=np.int64) for n in numels]
    if segments is None:
        if n_groups != len(numels):
            raise SegmentError("one group per tensor needs n_groups == n_tensors")
        for t, arr in enumerate(out):
            arr[:] = t
        return out
    for s in segments:
        if not (0 <= s.tensor_index < len(numels)):
            raise SegmentError(f"bad tensor index {s.tensor_index}")
        n = int(numels[s.tensor_index])
        if s.length <= 0 or s.start < 0 or s.start + s.length > n:
            raise SegmentError(f"segment {s} outside its tensor of {n} elements")
        if not (0 <= s.group_id < n_groups):
            raise SegmentError(f"group id {s.group_id} outside [0, {n_groups})")
        end = s.start + s.length
        if s.start % QBLOCK or (end % QBLOCK and end != n):
            raise SegmentError(f"segment {s} is not aligned to {QBLOCK}-element blocks")
        b0, b1 = s.start // QBLOCK, n_blocks(end)
        arr = out[s.tensor_index]
        if np.any(arr[b0:b1] >= 0):
            raise SegmentError(f"segment {s} overlaps another segment")
        arr[b0:b1] = s.group_id
    return out


def group_sumsq(block_sumsq: Sequence[np.ndarray], groups: Sequence[np.ndarray],
                n_groups: int):
    """Per-group sum of squares (fp64) and inverse Frobenius norm (fp32).

    ``inv[g] = 1 / (sqrt(S[g]) + 1e-7)`` -- the normalisation that turns the
    momentum into the Newton-Schulz input (section "What Exists", the
    ``..._and_normalize_groups_`` path).
    """
    S = np.zeros(n_groups, dtype=np.float64)
    for bs, gid in zip(block_sumsq, groups):
        bs = np.asarray(bs, dtype=np.float64)
        gid = np.asarray(gid)
        for g in range(n_groups):
            sel = gid == g
            if sel.any():
                S[g] += float(np.sum(bs[sel]))
    inv = (1.0 / (np.sqrt(S) + EPS)).astype(F32)
    return S, inv


def normalize_inplace(grad: np.ndarray, groups: np.ndarray, inv: np.ndarray,
                      grad_dtype: str = "bf16") -> np.ndarray:
    """Scale every block of a stored momentum by its group's inverse norm.

    This is the in-place normalisation of "What Exists"
    (``..._and_normalize_``): ``g <- store(float(g) * inv[group])`` in fp32
    with one rounding, blocks without a group left unchanged.
    """
    flat = np.asarray(grad).reshape(-1)
    numel = flat.size
    g32 = _pad_blocks(grad_to_f32(flat, grad_dtype), numel)
    gid = np.asarray(groups)
    scale = np.where(gid >= 0, np.asarray(inv, dtype=F32)[np.maximum(gid, 0)], F32(1.0)).astype(F32)
    scaled = (g32 * scale[:, None]).astype(F32)
    keep = gid < 0
    scaled[keep] = g32[keep]
    return f32_to_grad(scaled.reshape(-1)[:numel], grad_dtype)


def multi_update(q8s, absmaxes, grads, beta, *, grad_dtype="bf16", q8_kind="int8",
                 segments=None, n_groups=None, sr_seed: Optional[int] = None, sr_step: int = 0):
    """Update a list of tensors and reduce their norm groups.

    The multi-tensor form of "What Exists" (one call over many tensors, each
    gradient overwritten with the new momentum) with the grouped reduction of
    "Grouped QKV And Sharding".  With ``sr_seed`` set, requantisation is
    stochastic, tensor i drawing with tensor word i.  Returns
    ``(results, S, inv, groups)``.
    """
    results = [momentum_update(q, a, g, beta, grad_dtype=grad_dtype, q8_kind=q8_kind,
                               rounding=None if sr_seed is None else StochasticRounding(sr_seed, sr_step, i))
               for i, (q, a, g) in enumerate(zip(q8s, absmaxes, grads))]
    numels = [np.asarray(q).size for q in q8s]
    if n_groups is None:
        n_groups = len(numels) if segments is None else 1 + max(s.group_id for s in segments)
    groups = block_groups(numels, segments, n_groups)
    S, inv = group_sumsq([r.block_sumsq for r in results], groups, n_groups)
    return results, S, inv, groups
