"""MuonBP block-periodic quantized Muon step -- CPU oracle (test infrastructure only).

Source: "MuonBP: Faster Muon via Block-Periodic Orthogonalization",
section "整体框架" (the flowchart: update the local momentum; if
``t mod P != 0`` orthogonalise each block independently and step with
``eta_block``; otherwise orthogonalise the whole matrix and step with
``eta_full``) and section "关键设计" items 1-3 (a block is the shard one
tensor-parallel rank holds, ``(m/r) x (n/c)`` for an ``r x c`` tiling;
``P = 1`` is Muon and ``P -> infinity`` is BlockMuon; two learning rates).
The momentum update is the quantized codec of "Quantized Muon Momentum".

Readings taken:
* steps count from ``t = 1``; step ``t`` is a full step when
  ``t mod P == 0`` (``P = 0`` stands for "never", i.e. BlockMuon);
* the momentum update is the EMA codec (``oracle.codec``) on every step --
  the flowchart's ``M = mu M + G`` is not used because the quantized codec
  fixes the EMA form;
* on a block step every tile gets its own Frobenius norm and its own
  Newton-Schulz (each rank would normalise its shard locally); on a full
  step each matrix is one norm group;
* the Newton-Schulz output (fp64) is rounded to fp32 and then to bf16 and
  written over the gradient; the fp32 master weight takes
  ``W <- W - eta * U`` with one rounded product and one rounded difference;
* no extra shape factor is applied to ``eta`` (the page names an RMS-matching
  rule without giving it): the configured learning rates are final.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import codec, ns

F32 = np.float32


def is_full_step(t: int, P: int) -> bool:
    """``t mod P == 0``; ``P == 0`` means never (BlockMuon)."""
    if P < 0:
        raise ValueError("P must be >= 0")
    return P != 0 and t % P == 0


def tile_segments(rows: int, cols: int, tile_r: int, tile_c: int, tensor_index: int,
                  group_base: int):
    """Norm segments of an ``tile_r x tile_c`` tiling of a row-major matrix.

    Tile ``(i, j)`` covers rows ``[i R/r, (i+1) R/r)`` and columns
    ``[j C/c, (j+1) C/c)``; it is group ``group_base + i * c + j``.  With
    ``c == 1`` a tile is one contiguous run of whole rows and gives one
    segment; otherwise it gives one segment per row.  Segments must sit on
    256-element block boundaries ("Grouped QKV And Sharding"), so a
    column tiling needs tile widths that are multiples of 256.
    """
    if rows % tile_r or cols % tile_c:
        raise ValueError("the tiling must divide the matrix")
    th, tw = rows // tile_r, cols // tile_c
    segs = []
    for i in range(tile_r):
        for j in range(tile_c):
            g = group_base + i * tile_c + j
            if tile_c == 1:
                segs.append(codec.NormSegment(tensor_index, i * th * cols, th * cols, g))
                continue
            for r in range(i * th, (i + 1) * th):
                segs.append(codec.NormSegment(tensor_index, r * cols + j * tw, tw, g))
    return segs


@dataclass
class MatrixState:
    rows: int
    cols: int
    q8: np.ndarray        # flat codes
    absmax: np.ndarray    # fp32 [nb]
    weight: np.ndarray    # fp32 [rows, cols]


def muonbp_step(t: int, P: int, states, grads, beta: float, eta_full: float,
                eta_block: float, tile=(1, 8), iters: int = ns.ITERS,
                coeffs=ns.COEFFS, q8_kind: str = "int8"):
    """One optimizer step over a list of matrices.

    ``grads`` are bf16 bit patterns (flat or 2-D).  Returns
    ``(new_states, U_bits, info)`` where ``U_bits`` are the bf16 updates left
    in the gradient buffers and ``info`` holds the group sums.
    """
    full = is_full_step(t, P)
    tr, tc = tile
    results = [codec.momentum_update(s.q8, s.absmax, g, beta, grad_dtype="bf16", q8_kind=q8_kind)
               for s, g in zip(states, grads)]
    numels = [s.rows * s.cols for s in states]
    if full:
        segments, n_groups = None, len(states)
    else:
        segments, n_groups = [], 0
        for k, s in enumerate(states):
            segments += tile_segments(s.rows, s.cols, tr, tc, k, n_groups)
            n_groups += tr * tc
    groups = codec.block_groups(numels, segments, n_groups)
    S, inv = codec.group_sumsq([r.block_sumsq for r in results], groups, n_groups)

    new_states, U_bits = [], []
    gbase = 0
    for k, (s, r) in enumerate(zip(states, results)):
        M = codec.f32_from_bf16_bits(r.grad).reshape(s.rows, s.cols).astype(np.float64)
        U = np.empty_like(M)
        if full:
            U[:] = ns.newton_schulz(M, inv_norm=float(inv[k]), iters=iters, coeffs=coeffs)
        else:
            th, tw = s.rows // tr, s.cols // tc
            for i in range(tr):
                for j in range(tc):
                    g = gbase + i * tc + j
                    blk = M[i * th:(i + 1) * th, j * tw:(j + 1) * tw]
                    U[i * th:(i + 1) * th, j * tw:(j + 1) * tw] = ns.newton_schulz(
                        blk, inv_norm=float(inv[g]), iters=iters, coeffs=coeffs)
            gbase += tr * tc
        ub = codec.bf16_bits_from_f32(U.astype(F32))
        u32 = codec.f32_from_bf16_bits(ub).reshape(s.rows, s.cols)
        eta = F32(eta_full if full else eta_block)
        W = (s.weight.astype(F32) - (eta * u32).astype(F32)).astype(F32)
        new_states.append(MatrixState(s.rows, s.cols, r.q8, r.absmax, W))
        U_bits.append(ub.reshape(s.rows, s.cols))
    return new_states, U_bits, {"full": full, "S": S, "inv": inv, "n_groups": n_groups}
