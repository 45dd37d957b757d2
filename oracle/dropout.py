"""Dropout on the attention probabilities, with a counter-based generator so that the backward can
regenerate the forward's mask ("dropout RNG" and "dropout replay"; FlashAttention：让精确注意力
服从内存层次, the list of production semantics after the CPU reference and the validation list in
its numerics section).

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py``; nothing in the product path imports it, and it shares no code with the CUDA
library (which implements the same published generator on its own).

The pages name the feature and ask that forward, backward and the replay be tested; they fix no
generator, mask layout or rate encoding.  The reading taken here:

* Generator: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC 2011): a 128-bit counter and a 64-bit key; ten rounds, each multiplying counter
  words 0 and 2 by two fixed odd constants into 64-bit products, and xoring the high halves
  with the other counter words and the key; the key is advanced by two Weyl constants between
  rounds.
* One call covers a 4 x 4 block of the score matrix of one (b, h) slice: counter =
  (j // 4, i // 4, b * H + h, offset), key = (seed mod 2^32, seed // 2^32).  Output word
  (i mod 4), byte (j mod 4) is the 8-bit uniform u(i, j) of element (i, j).
* Element (i, j) is kept iff u(i, j) < k8, where k8 = round((1 - p) * 256) in [0, 256] is the
  keep threshold: the keep probability is exactly k8 / 256.  Kept probabilities are scaled by
  256 / k8 (inverted dropout); with k8 = 0 everything is dropped and the output is zero.
* Dropout acts on P after the softmax: O = (P * M * 256/k8) V; the softmax statistic (LSE) is
  that of the undropped scores.  In the backward, dV = (P * M * 256/k8)^T dO and
  dP = (dO V^T) * M * 256/k8, with D and dS as without dropout (D = rowsum(dO * O) still equals
  sum_j P_ij dP_ij).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57      # Philox4x32 round multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85      # Weyl increments of the key
MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32-10 on arrays: counter uint [..., 4], key uint [..., 2] -> uint32 [..., 4]."""
    c = np.asarray(counter, dtype=np.uint64) & MASK32
    k = np.asarray(key, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = (c[..., n].copy() for n in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    for r in range(10):
        if r > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = np.uint64(M0) * c0          # < 2^64: exact in uint64
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def keep_threshold(p: float) -> int:
    """k8 = round((1 - p) * 256), clipped to [0, 256]: the keep probability is k8 / 256."""
    return int(min(256, max(0, int(np.rint((1.0 - float(p)) * 256.0)))))


def uniforms(rows, cols, bh: int, seed: int, offset: int) -> np.ndarray:
    """8-bit uniforms u(i, j) (uint8 [len(rows), len(cols)]) of slice index bh = b * H + h."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    I, J = np.meshgrid(rows, cols, indexing="ij")
    ctr = np.stack([J >> 2, I >> 2, np.full_like(I, bh), np.full_like(I, offset)], axis=-1)
    key = np.array([seed & MASK32, (seed >> 32) & MASK32], dtype=np.uint64)
    words = philox4x32_10(ctr, np.broadcast_to(key, ctr.shape[:-1] + (2,)))
    w = np.take_along_axis(words, (I & 3)[..., None], axis=-1)[..., 0]
    return ((w >> (8 * (J & 3)).astype(np.uint32)) & 0xFF).astype(np.uint8)


def keep_mask(rows, cols, bh: int, seed: int, offset: int, k8: int) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: which probabilities survive dropout."""
    return uniforms(rows, cols, bh, seed, offset).astype(np.int64) < int(k8)


def scale_of(k8: int) -> float:
    """Factor applied to the kept probabilities (0 when everything is dropped)."""
    return 256.0 / k8 if k8 > 0 else 0.0
