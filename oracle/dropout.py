"""Attention dropout in fp64 — TEST INFRASTRUCTURE ONLY.

The FlashAttention review page ("长上下文能力：FlashAttention vs.
RingAttention", FlashAttention-1 核心优化, 算子融合) names dropout among the
operations fused with the matmuls, the mask and the softmax.  Semantics
(inverted dropout on the attention probabilities): with P the softmax of the
scores and Z_ij in {0, 1} drawn independently with P(Z = 1) = k,

    O = (P * Z / k) V,    LSE unchanged (computed from P).

Backward, with dP~ = dO V^T the gradient of the dropped probabilities:

    dV = (P * Z / k)^T dO,   D_i = sum_j (P*Z/k)_ij dP~_ij = dO_i . O_i,
    dS = P * (Z/k * dP~ - D),  dQ = tau dS K,  dK = tau dS^T Q.

Random bits: Philox4x32-10, the counter-based generator of Salmon, Moraes,
Dror and Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011),
written here from its definition: ten rounds, each multiplying two of the four
32-bit counter words by fixed odd constants and mixing the high and low product
halves with the other words and the key; the key gains a Weyl increment
between rounds.  One call covers query head h, global query row i and 16
consecutive keys of the row's segment (j counted from the segment's first
key): counter = (j // 16, i, h, 0), key = (seed low 32
bits, seed high 32 bits); element j uses byte j % 4 of output word (j % 16) // 4.
It is kept when that byte is >= t = floor(256 p + 1/2), p the drop
probability taken as a float32 and t capped at 255, so k = (256 - t) / 256
and the kept values are scaled by 256 / (256 - t).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57  # round multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85  # key increments (Weyl sequence)
MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """counter: uint [..., 4]; key: (k0, k1).  Returns uint32 [..., 4]."""
    c = [np.asarray(counter, dtype=np.uint64)[..., t] & MASK32 for t in range(4)]
    k0, k1 = np.uint64(int(key[0]) & MASK32), np.uint64(int(key[1]) & MASK32)
    for r in range(10):
        if r > 0:
            k0 = (k0 + np.uint64(W0)) & np.uint64(MASK32)
            k1 = (k1 + np.uint64(W1)) & np.uint64(MASK32)
        p0 = c[0] * np.uint64(M0)  # full 64-bit products of 32-bit values
        p1 = c[2] * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK32)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack(c, axis=-1).astype(np.uint32)


def drop_threshold(p: float) -> int:
    t = int(np.floor(256.0 * float(np.float32(p)) + 0.5))
    return min(255, max(0, t))


def keep_mask(seed: int, p: float, head: int, rows, cols) -> np.ndarray:
    """Z for global query rows `rows` x keys `cols` (indices within the rows'
    segment) of query head `head` (bool)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    groups = np.unique(cols // 16)
    ctr = np.zeros((rows.size, groups.size, 4), dtype=np.uint64)
    ctr[..., 0] = groups[None, :]
    ctr[..., 1] = rows[:, None]
    ctr[..., 2] = head
    words = philox4x32_10(ctr, (seed & MASK32, (seed >> 32) & MASK32))  # [rows, groups, 4]
    g = np.searchsorted(groups, cols // 16)
    w = words[:, g, (cols % 16) // 4]  # [rows, cols]
    byte = (w >> (8 * (cols % 4))[None, :].astype(np.uint32)) & 0xFF
    return byte >= drop_threshold(p)


def keep_scale(p: float) -> float:
    """1 / k, the factor applied to the kept probabilities."""
    return 256.0 / (256 - drop_threshold(p))


def scaled_keep(dropout, head: int, rows, cols) -> np.ndarray:
    """Z / k (fp64) for global query rows x segment key columns of one head;
    `dropout` is (seed, p)."""
    seed, p = dropout
    return keep_mask(seed, p, head, rows, cols) * keep_scale(p)
