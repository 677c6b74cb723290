"""Philox4x32-10 counter-based generator -- CPU oracle (test infrastructure only).

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3" (SC'11), the Philox-4x32 bijection with 10
rounds.  A round maps the counter (c0, c1, c2, c3) under the key (k0, k1) to

    (hi(M1 c2) ^ c1 ^ k0,  lo(M1 c2),  hi(M0 c0) ^ c3 ^ k1,  lo(M0 c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57 and hi/lo the two 32-bit halves of the
64-bit product; between rounds the key is bumped by the Weyl constants
(0x9E3779B9, 0xBB67AE85) modulo 2^32.

Use in the stochastic requantisation (a reading: the page only says that
stochastic rounding is not implemented yet): the key is the 64-bit seed
(low word, high word); element e of tensor i at step t draws word (e mod 4)
of the block for counter (e // 4 mod 2^32, e // 2^34, i, t mod 2^32); its top
24 bits give the uniform u = (word >> 8) * 2^-24 in [0, 1).
"""

from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(counter: np.ndarray, key) -> np.ndarray:
    """Philox4x32-10 of each row of ``counter`` ([N, 4] uint32) under ``key``
    (two uint32 words); returns [N, 4] uint32."""
    ctr = np.asarray(counter, dtype=np.uint64).reshape(-1, 4)
    c0, c1, c2, c3 = (ctr[:, i].copy() for i in range(4))
    k0, k1 = np.uint64(int(key[0]) & _MASK), np.uint64(int(key[1]) & _MASK)
    m0, m1, mask = np.uint64(M0), np.uint64(M1), np.uint64(_MASK)
    for r in range(10):
        if r > 0:
            k0 = np.uint64((int(k0) + W0) & _MASK)
            k1 = np.uint64((int(k1) + W1) & _MASK)
        p0 = m0 * c0          # both factors < 2^32: exact in uint64
        p1 = m1 * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & mask,
                          (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & mask)
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def rounding_uniforms(numel: int, seed: int, step: int, tensor_index: int) -> np.ndarray:
    """The uniforms u in [0, 1) (fp64, multiples of 2^-24) of a tensor's
    ``numel`` elements for the stochastic requantisation."""
    nblk = (numel + 3) // 4
    j = np.arange(nblk, dtype=np.uint64)
    ctr = np.empty((nblk, 4), dtype=np.uint64)
    ctr[:, 0] = j & np.uint64(_MASK)
    ctr[:, 1] = j >> np.uint64(32)
    ctr[:, 2] = np.uint64(tensor_index & _MASK)
    ctr[:, 3] = np.uint64(step & _MASK)
    words = philox4x32_10(ctr, (seed & _MASK, (seed >> 32) & _MASK)).reshape(-1)[:numel]
    return (words >> np.uint32(8)).astype(np.float64) * 2.0 ** -24
