"""Seeded synthetic workloads for the quantized Muon step.

Shapes, value distributions, norm-group layouts and hyper-parameters of the
five synthetic workloads, plus seeded generators for their gradients,
states and master weights.  This module holds none of the method's
arithmetic: it only draws inputs.  Both the CUDA library's tests/bench and the
CPU oracle's tests consume what it produces (generated once, copied to the
other side), so the two never disagree about inputs.

Seeds: the gradient of step ``s`` of workload ``k`` uses ``1000 * k + s``;
master weights use ``1000 * k + 999``.  Generators run on whatever device
they are given (CUDA for large workloads); torch's CPU and CUDA generators
produce different streams, so parity tests generate once and copy.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

COEFFS = (3.4445, -4.7750, 2.0315)


@dataclass(frozen=True)
class Matrix:
    name: str
    rows: int
    cols: int

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Segment:
    tensor_index: int
    start: int
    length: int
    group_id: int


@dataclass
class Workload:
    key: int
    name: str
    matrices: List[Matrix]
    grad_dist: str                 # "normal_1e-3" | "rowscale_lognormal1" | "outliers" | "colscale_lognormal1.5"
    q8_kind: str = "int8"
    beta: float = 0.95
    steps: int = 10
    segments: Optional[List[Segment]] = None   # None: one norm group per matrix
    n_groups: Optional[int] = None
    ns_slices: Optional[List[Tuple[int, int, int]]] = None  # (tensor, row0, rows) NS problems; None: whole matrices
    ns: bool = True
    P: int = 1
    tile: Tuple[int, int] = (1, 1)
    eta_full: float = 0.02
    eta_block: float = 0.02
    iters: int = 5
    coeffs: Tuple[float, float, float] = COEFFS
    carrier: bool = False
    notes: str = ""

    @property
    def numel(self) -> int:
        return sum(m.numel for m in self.matrices)

    @property
    def groups(self) -> int:
        return len(self.matrices) if self.segments is None else int(self.n_groups)


def _decoder_2048_24() -> List[Matrix]:
    # per layer q,k,v,o 2048x2048; gate,up 8192x2048; down 2048x8192 -- repeated
    # and cut at 24 matrices (3 full layers + q,k,v of a fourth)
    layer = [("q", 2048, 2048), ("k", 2048, 2048), ("v", 2048, 2048), ("o", 2048, 2048),
             ("gate", 8192, 2048), ("up", 8192, 2048), ("down", 2048, 8192)]
    out = []
    i = 0
    while len(out) < 24:
        n, r, c = layer[i % 7]
        out.append(Matrix(f"l{i // 7}.{n}", r, c))
        i += 1
    return out


def _llama8b_layers(n_layers: int = 4) -> List[Matrix]:
    layer = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
             ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
    return [Matrix(f"l{l}.{n}", r, c) for l in range(n_layers) for (n, r, c) in layer]


def _qkv_mlp() -> Tuple[List[Matrix], List[Segment], List[Tuple[int, int, int]]]:
    mats = [Matrix("qkv", 12288, 4096)]
    mats += [Matrix(f"mlp{i}.up", 14336, 4096) for i in range(4)]
    mats += [Matrix(f"mlp{i}.down", 4096, 14336) for i in range(4)]
    third = 4096 * 4096
    segs = [Segment(0, g * third, third, g) for g in range(3)]
    segs += [Segment(1 + i, 0, mats[1 + i].numel, 3 + i) for i in range(8)]
    slices = [(0, 0, 4096), (0, 4096, 4096), (0, 8192, 4096)] + [(1 + i, 0, mats[1 + i].rows) for i in range(8)]
    return mats, segs, slices


def get(key: int, q8_kind: Optional[str] = None) -> Workload:
    """The five synthetic workloads, numbered 1..5; ``q8_kind`` ("int8" or
    "uint8") replaces the workload's code kind (the grouped workload 3 names
    both)."""
    w = _get(key)
    if q8_kind is not None:
        if q8_kind not in ("int8", "uint8"):
            raise ValueError(q8_kind)
        w.q8_kind = q8_kind
    return w


def _get(key: int) -> Workload:
    if key == 1:
        return Workload(1, "one 512x512 matrix, grad N(0,1e-3^2), 3 steps, Frobenius normalise + 5 NS iterations",
                        [Matrix("w", 512, 512)], "normal_1e-3", steps=3)
    if key == 2:
        return Workload(2, "24 matrices of a 2048-hidden decoder, per-tensor norm, update only",
                        _decoder_2048_24(), "rowscale_lognormal1", steps=10, ns=False)
    if key == 3:
        mats, segs, slices = _qkv_mlp()
        return Workload(3, "fused QKV 12288x4096 (3 row groups) + 8 MLP matrices, grouped normalise + 5 NS iterations",
                        mats, "outliers", steps=10, segments=segs, n_groups=11, ns_slices=slices)
    if key == 4:
        return Workload(4, "MuonBP on 4 Llama-8B layers: 1x8 column tiles, P=5, eta_full=0.02, eta_block=0.02/sqrt(8)",
                        _llama8b_layers(4), "rowscale_lognormal1", steps=20, P=5, tile=(1, 8),
                        eta_full=0.02, eta_block=0.02 / math.sqrt(8.0))
    if key == 5:
        return Workload(5, "MXFP8 carrier on 4 Llama-8B layers: E4M3 payload + E8M0 scale per 32 row elements, full NS",
                        _llama8b_layers(4), "colscale_lognormal1.5", steps=10, carrier=True)
    raise KeyError(key)


def grad_seed(key: int, step: int) -> int:
    return 1000 * key + step


def make_grad(w: Workload, index: int, step: int, device="cpu", dtype=torch.bfloat16,
              matrix: Optional[Matrix] = None) -> torch.Tensor:
    """The gradient of matrix ``index`` at ``step`` (row-major, ``dtype``)."""
    m = matrix if matrix is not None else w.matrices[index]
    g = torch.Generator(device=device)
    g.manual_seed(grad_seed(w.key, step) * 1009 + index)
    shape = (m.rows, m.cols)
    if w.grad_dist == "normal_1e-3":
        x = torch.randn(shape, generator=g, device=device) * 1e-3
    elif w.grad_dist == "rowscale_lognormal1":
        z = torch.randn(shape, generator=g, device=device)
        s = torch.exp(torch.randn((m.rows, 1), generator=g, device=device))
        x = z * s
    elif w.grad_dist == "colscale_lognormal1.5":
        z = torch.randn(shape, generator=g, device=device)
        s = torch.exp(1.5 * torch.randn((1, m.cols), generator=g, device=device))
        x = z * s
    elif w.grad_dist == "outliers":
        x = torch.randn(shape, generator=g, device=device)
        hit = torch.rand(shape, generator=g, device=device) < 1e-3
        x = torch.where(hit, x * 100.0, x)
    else:
        raise ValueError(w.grad_dist)
    return x.to(dtype).contiguous()


def make_weight(w: Workload, index: int, device="cpu") -> torch.Tensor:
    m = w.matrices[index]
    g = torch.Generator(device=device)
    g.manual_seed((1000 * w.key + 999) * 1009 + index)
    return (torch.randn((m.rows, m.cols), generator=g, device=device) * 0.02).contiguous()


def zero_state(m: Matrix, q8_kind: str = "int8", device="cpu"):
    """A fresh quantized state: zero codes (offset 128 for uint8) and zero absmax."""
    nb = (m.numel + 255) // 256
    if q8_kind == "int8":
        q = torch.zeros(m.numel, dtype=torch.int8, device=device)
    else:
        q = torch.full((m.numel,), 128, dtype=torch.uint8, device=device)
    return q, torch.zeros(nb, dtype=torch.float32, device=device)


def random_state(m: Matrix, seed: int, q8_kind: str = "int8", device="cpu"):
    """A non-trivial state: random codes in [-127, 127] and log-uniform absmax."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nb = (m.numel + 255) // 256
    q = torch.randint(-127, 128, (m.numel,), generator=g, device=device, dtype=torch.int32)
    a = torch.exp(torch.empty(nb, device=device).uniform_(-9.0, 3.0, generator=g)).float()
    if q8_kind == "int8":
        return q.to(torch.int8), a
    return (q + 128).to(torch.uint8), a


def scaled(w: Workload, factor: int) -> Workload:
    """A copy of a workload with every matrix dimension divided by ``factor``
    (rounded up to a multiple of 256) -- the same structure at a size the
    oracle finishes in seconds."""
    def sh(x):
        return max(256, ((x // factor + 255) // 256) * 256)
    mats = [Matrix(m.name, sh(m.rows), sh(m.cols)) for m in w.matrices]
    out = Workload(**{**w.__dict__, "matrices": mats})
    if w.segments is not None:
        # re-derive row-third groups for the fused QKV and one group per other matrix
        segs = []
        q = mats[0]
        third_rows = q.rows // 3
        for g in range(3):
            segs.append(Segment(0, g * third_rows * q.cols, third_rows * q.cols, g))
        for i, m in enumerate(mats[1:]):
            segs.append(Segment(1 + i, 0, m.numel, 3 + i))
        out.segments = segs
        out.ns_slices = [(0, g * third_rows, third_rows) for g in range(3)] + \
                        [(1 + i, 0, m.rows) for i, m in enumerate(mats[1:])]
    return out
