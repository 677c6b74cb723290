"""4-bit GRASP momentum state -- CPU oracle (test infrastructure only).

Source: "4-bit-Muon-GRASP" (zij math notes), the update equations and the
grid-quantisation formula on that page.  The momentum of an rows x cols matrix
is held as a rank-k factor P R^T (P: rows x k, R: cols x k, 8-bit) plus a
residual (4-bit); one warm-started power iteration refreshes the factor every
step, and every piece is stored with grid quantisation, each entry scaled by
the smaller of its row and column maxima inside its block.

Readings taken where the page is silent (the parameters are arguments):

* rank k = 8 and grid block s = 64 by default; blocks at the matrix edge are
  partial and their maxima run over the elements that exist;
* QUANT_b is symmetric and uniform with L = 2^(b-1) - 1 levels a side (7 for
  the residual, 127 for P and R): with r_i, c_j the block's row and column
  maxima of |x| and d = min(r_i, c_j), ``q = clamp(rint(x * fl(L / d)), -L,
  L)`` in fp32 (ties to even, q = 0 where d = 0) and the value read back is
  ``q * fl(d / L)``; the scales are stored as the fp32 maxima;
* P and R are grid-quantised in blocks of s rows by all k columns;
* the momentum step is the page's ``M_t = mu M_{t-1} + g_t`` in fp32, one
  rounding per operation, with ``M_{t-1} = res + P R^T`` reconstructed as
  ``fl(res + sum_l fl(p_il r_jl))`` summed over l in order (no fused
  multiply-add); M_t is stored in bf16 over the gradient and every later use
  (power iteration, residual, Newton-Schulz) reads that bf16 value;
* ``Q_t = ColNorm(R_{t-1})`` divides each column of the dequantised R by its
  2-norm (a zero column stays zero); ``P_t = Orthogonalize(M_t Q_t)`` is the
  orthonormal factor of the thin QR decomposition whose triangular factor has
  a positive diagonal; ``R_t = M_t^T P_t``; the residual ``M_t - P_t R_t^T``
  uses these unquantised P_t and R_t, and the three are quantised afterwards;
* the power iteration runs in fp64 here;
* at the first step the state is zero except R, which the caller seeds
  (a fixed Gaussian: the warm start has to start somewhere).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import codec

F32 = np.float32


def grid_quantize(x: np.ndarray, bits: int, s_rows: int, s_cols: int):
    """Grid quantisation of a 2-D fp32 array in blocks of s_rows x s_cols.

    Returns (codes int8 [R, C], rmax fp32 [nbc, R], cmax fp32 [nbr, C]):
    rmax[bj, i] is row i's max |x| inside column block bj, cmax[bi, j] column
    j's max |x| inside row block bi."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    L = F32(2 ** (bits - 1) - 1)
    nbr, nbc = -(-R // s_rows), -(-C // s_cols)
    a = np.abs(x)
    rmax = np.zeros((nbc, R), F32)
    cmax = np.zeros((nbr, C), F32)
    for bj in range(nbc):
        rmax[bj] = a[:, bj * s_cols:(bj + 1) * s_cols].max(axis=1)
    for bi in range(nbr):
        cmax[bi] = a[bi * s_rows:(bi + 1) * s_rows, :].max(axis=0)
    d = _block_min(rmax, cmax, R, C, s_rows, s_cols)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d == 0, F32(0.0), (L / np.where(d == 0, F32(1.0), d)).astype(F32)).astype(F32)
        q = np.rint((x * sc).astype(F32))
    q = np.clip(np.where(np.isnan(q), 0.0, q), -L, L).astype(np.int8)
    return q, rmax, cmax


def _block_min(rmax, cmax, R, C, s_rows, s_cols):
    """d_ij = min(row max of i in j's column block, column max of j in i's row block)."""
    rb = np.repeat(rmax.T, s_cols, axis=1)[:, :C]          # [R, C]: rmax[j // s_cols, i]
    cb = np.repeat(cmax, s_rows, axis=0)[:R, :]            # [R, C]: cmax[i // s_rows, j]
    return np.minimum(rb, cb).astype(F32)


def grid_dequantize(q: np.ndarray, rmax: np.ndarray, cmax: np.ndarray, bits: int, s_rows: int, s_cols: int):
    R, C = q.shape
    L = F32(2 ** (bits - 1) - 1)
    d = _block_min(rmax, cmax, R, C, s_rows, s_cols)
    step = (d / L).astype(F32)
    return (q.astype(F32) * step).astype(F32)


def pack4(q: np.ndarray) -> np.ndarray:
    """4-bit codes, two per byte: column 2c in the low nibble, 2c + 1 in the
    high one, each as q + 8 (offset binary)."""
    q = np.asarray(q, dtype=np.int16)
    R, C = q.shape
    if C % 2:
        raise ValueError("4-bit packing needs an even number of columns")
    u = (q + 8).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack4(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    lo = (b & 0x0F).astype(np.int16) - 8
    hi = (b >> 4).astype(np.int16) - 8
    out = np.empty((b.shape[0], b.shape[1] * 2), np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


@dataclass
class GraspState:
    res: np.ndarray        # uint8 [rows, cols / 2] packed 4-bit residual codes
    res_rmax: np.ndarray   # fp32 [ceil(cols / s), rows]
    res_cmax: np.ndarray   # fp32 [ceil(rows / s), cols]
    p: np.ndarray          # int8 [rows, k]
    p_rmax: np.ndarray     # fp32 [1, rows]
    p_cmax: np.ndarray     # fp32 [ceil(rows / s), k]
    r: np.ndarray          # int8 [cols, k]
    r_rmax: np.ndarray     # fp32 [1, cols]
    r_cmax: np.ndarray     # fp32 [ceil(cols / s), k]


def initial_state(rows: int, cols: int, r0: np.ndarray, k: int = 8, s: int = 64) -> GraspState:
    """Zero residual and P; R holds the quantised warm start ``r0`` (cols x k)."""
    rq, rr, rc = grid_quantize(np.asarray(r0, F32), 8, s, k)
    nbc, nbr = -(-cols // s), -(-rows // s)
    return GraspState(res=np.full((rows, cols // 2), 0x88, np.uint8),
                      res_rmax=np.zeros((nbc, rows), F32), res_cmax=np.zeros((nbr, cols), F32),
                      p=np.zeros((rows, k), np.int8), p_rmax=np.zeros((1, rows), F32),
                      p_cmax=np.zeros((nbr, k), F32), r=rq, r_rmax=rr, r_cmax=rc)


def dequantize_parts(st: GraspState, s: int = 64):
    k = st.p.shape[1]
    res = grid_dequantize(unpack4(st.res), st.res_rmax, st.res_cmax, 4, s, s)
    p = grid_dequantize(st.p, st.p_rmax, st.p_cmax, 8, s, k)
    r = grid_dequantize(st.r, st.r_rmax, st.r_cmax, 8, s, k)
    return res, p, r


def reconstruct(res: np.ndarray, p: np.ndarray, r: np.ndarray) -> np.ndarray:
    """``fl(res + sum_l fl(p_il r_jl))``, the sum over l left to right in fp32."""
    acc = np.zeros(res.shape, F32)
    for l in range(p.shape[1]):
        acc = (acc + (p[:, l:l + 1] * r[:, l][None, :]).astype(F32)).astype(F32)
    return (res + acc).astype(F32)


def orthonormal_factor(y: np.ndarray) -> np.ndarray:
    """Q factor of the thin QR of y (fp64) with the triangular factor's
    diagonal made positive."""
    qf, rf = np.linalg.qr(np.asarray(y, np.float64))
    sgn = np.where(np.diag(rf) < 0, -1.0, 1.0)
    return qf * sgn[None, :]


@dataclass
class GraspStep:
    state: GraspState
    m_bits: np.ndarray   # uint16 bf16 bits [rows, cols]: M_t as stored over the gradient
    m_prev: np.ndarray   # fp32 reconstruction of M_{t-1}
    q: np.ndarray        # fp64 [cols, k] ColNorm(R_{t-1})
    y: np.ndarray        # fp64 [rows, k] M_t Q_t
    p: np.ndarray        # fp64 [rows, k] P_t
    r: np.ndarray        # fp64 [cols, k] R_t
    res: np.ndarray      # fp64 [rows, cols] M_t - P_t R_t^T


def grasp_step(st: GraspState, grad_bits: np.ndarray, mu: float, s: int = 64) -> GraspStep:
    """One GRASP momentum step of one matrix (page equations, in order)."""
    rows, k = st.p.shape
    cols = st.r.shape[0]
    res, p_old, r_old = dequantize_parts(st, s)
    m_prev = reconstruct(res, p_old, r_old)                                  # M_{t-1}
    g = codec.f32_from_bf16_bits(np.asarray(grad_bits).reshape(rows, cols))
    m = ((F32(mu) * m_prev).astype(F32) + g).astype(F32)                     # M_t = mu M_{t-1} + g_t
    m_bits = codec.bf16_bits_from_f32(m.reshape(-1)).reshape(rows, cols)
    mt = codec.f32_from_bf16_bits(m_bits).astype(np.float64)                 # the stored M_t
    r64 = r_old.astype(np.float64)
    nrm = np.linalg.norm(r64, axis=0)
    q = np.where(nrm[None, :] > 0, r64 / np.where(nrm == 0, 1.0, nrm)[None, :], 0.0)   # ColNorm(R_{t-1})
    y = mt @ q
    p = orthonormal_factor(y)                                                # P_t
    r = mt.T @ p                                                             # R_t
    resid = mt - p @ r.T                                                     # M_res,t
    rq, rr, rc = grid_quantize(resid.astype(F32), 4, s, s)
    pq, pr, pc = grid_quantize(p.astype(F32), 8, s, k)
    q8, r8r, r8c = grid_quantize(r.astype(F32), 8, s, k)
    new = GraspState(res=pack4(rq), res_rmax=rr, res_cmax=rc, p=pq, p_rmax=pr, p_cmax=pc,
                     r=q8, r_rmax=r8r, r_cmax=r8c)
    return GraspStep(state=new, m_bits=m_bits, m_prev=m_prev, q=q, y=y, p=p, r=r, res=resid)
