"""Helpers shared by the GPU parity tests (device <-> oracle representations)."""

import numpy as np
import torch

TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def to_oracle_grad(t: torch.Tensor, dtype: str) -> np.ndarray:
    """A device gradient as the oracle stores it (bf16 as uint16 bits)."""
    t = t.detach().contiguous().cpu().reshape(-1)
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "f16":
        return t.numpy().copy()
    return t.numpy().astype(np.float32).copy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def min_row_cos(a: np.ndarray, b: np.ndarray) -> float:
    na = np.linalg.norm(a, axis=1)
    nb = np.linalg.norm(b, axis=1)
    keep = nb > 0
    return float(np.min(np.sum(a[keep] * b[keep], axis=1) / (na[keep] * nb[keep])))


def ulp_diff_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> int:
    """Largest distance in bf16 ulps between two arrays of bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return int(np.max(np.abs(ordered(a_bits) - ordered(b_bits)))) if a_bits.size else 0


def random_grad(n: int, dtype: str, seed: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nb = (n + 255) // 256
    scale = torch.exp(torch.empty(nb, device=device).uniform_(-8.0, 4.0, generator=g)).repeat_interleave(256)[:n]
    x = torch.randn(n, generator=g, device=device) * scale
    x[torch.rand(n, generator=g, device=device) < 0.02] = 0.0
    return x.to(TORCH_DT[dtype]).contiguous()


GUARD = 4096          # guard bytes on each side of a buffer (keeps 256-byte alignment)
GUARD_BYTE = 0xA5


class Guarded:
    """A device tensor of ``shape``/``dtype`` inside a larger byte buffer whose
    GUARD bytes before and after hold a fixed pattern; ``check()`` asserts the
    pattern is intact (a write outside the tensor shows up there)."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= int(s)
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((self.nbytes + 2 * GUARD,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def check(self, what=""):
        lo, hi = self.raw[:GUARD], self.raw[GUARD + self.nbytes:]
        assert bool((lo == GUARD_BYTE).all()) and bool((hi == GUARD_BYTE).all()), f"guard bytes overwritten {what}"


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 values rounded to bf16 (nearest even) and back."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy() \
        .astype(np.float64)


def one_iteration_reference(M: np.ndarray, coeffs, inv: float) -> np.ndarray:
    """One Newton-Schulz iteration with the engine's rounding points: A and the
    polynomial B = a I + b A + c A A (the a X term folded into B's diagonal)
    are stored in bf16, the update is the single product B X; everything else
    is fp64."""
    a, b, c = coeffs
    X = M * inv
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    A = bf16_round(X @ X.T)
    B = bf16_round(a * np.eye(A.shape[0]) + b * A + c * (A @ A))
    out = B @ X
    return out.T if tall else out
