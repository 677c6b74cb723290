"""Quintic Newton-Schulz orthogonalisation -- fp64 CPU oracle (test infrastructure only).

Sources:
* "NVIDIA impulsa optimizadores avanzados para mejorar el entrenamiento de
  LLMs con Megatron", section "Newton-Schulz distribuido" (each iteration is
  three matrix products) and section "SYRK y reducción fusionada" (the first
  two products are symmetric);
* "MuonBP: Faster Muon via Block-Periodic Orthogonalization", section
  "关键设计" item 1 (per-iteration cost ``2(2nm^2 + m^3)`` for an ``m x n``
  matrix with ``m <= n``);
* "Quantized Muon Momentum", sections "What Exists" and "Local Megatron
  Integration" (the Newton-Schulz input is the momentum after Frobenius
  normalisation, per norm group).

Readings taken (the pages do not print the iteration):
* one iteration is ``A = X X^T``, ``B = b A + c A A``, ``X <- a X + B X``,
  with ``(a, b, c) = (3.4445, -4.7750, 2.0315)`` and 5 iterations unless
  given;
* a matrix with more rows than columns is transposed first (so the Gram
  matrix is the smaller one) and transposed back at the end;
* ``X_0 = inv_norm * M`` where ``inv_norm`` comes from the momentum update's
  group sums.

Everything is fp64; matrix products use numpy's ``@``.
"""

from __future__ import annotations

import numpy as np

COEFFS = (3.4445, -4.7750, 2.0315)
ITERS = 5


def ns_flops(rows: int, cols: int, iters: int = ITERS) -> float:
    """Algorithmic FLOPs of ``iters`` iterations: ``2(2nm^2 + m^3)`` each."""
    m, n = min(rows, cols), max(rows, cols)
    return float(iters) * 2.0 * (2.0 * n * m * m + float(m) ** 3)


def newton_schulz(M: np.ndarray, inv_norm=None, iters: int = ITERS, coeffs=COEFFS) -> np.ndarray:
    """Orthogonalise ``M`` (any 2-D shape) in fp64.

    ``inv_norm=None`` normalises by ``1 / (||M||_F + 1e-7)``; otherwise the
    given scalar (the group inverse norm) is applied.
    """
    a, b, c = (float(v) for v in coeffs)
    X = np.asarray(M, dtype=np.float64)
    if inv_norm is None:
        inv_norm = 1.0 / (np.linalg.norm(X) + 1e-7)
    X = X * float(inv_norm)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    for _ in range(iters):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    if transposed:
        X = X.T
    return np.ascontiguousarray(X)

