"""Dropout keep-mask of the attention oracle (test infrastructure only).

Imported by the tests, the smoke check and the bench's CPU-baseline leg; the
product path never imports it and it shares no code with the CUDA library.

The pages name dropout as one of the stages of attention that the method
fuses into its single kernel ("Matmul / Mask / Softmax / Dropout / Matmul",
GPT-2 time-breakdown figure caption on the aggregator page) and note that the
memory footprint does not depend on it. They fix neither the generator nor
how a draw becomes a keep decision, so the following reading is taken:

  * Inverted dropout on the attention probabilities: Pd = P * Z / (1 - p'),
    O = Pd V, with Z_ij in {0, 1}. LSE is that of the undropped scores.
  * The draws come from Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror,
    D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, the
    Philox-4x32 bijection with 10 rounds), a counter-based generator, so the
    backward pass regenerates the same Z from indices instead of storing it.
  * Key = (seed mod 2^32, seed div 2^32). Element (b, h, i, j) of a problem
    with H heads draws from counter (j div 16, i, b*H + h, offset): one Philox
    block of four 32-bit words gives 16 bytes, byte e (bits 8(e mod 4) ..
    8(e mod 4)+7 of word e div 4) belonging to key j = 16 (j div 16) + e.
  * The drop probability is taken in steps of 1/256: t = round(256 p), capped
    at 255; an element is kept iff its byte >= t (so p' = t / 256) and kept
    entries are scaled by 256 / (256 - t) = 1 / (1 - p'), which keeps
    E[Z / (1 - p')] = 1 exactly.

Pins (tests/test_oracle_dropout.py): the generator against the cuRAND host
Philox4_32_10 generator (a library routine), the byte and keep statistics,
p = 0 reducing to plain attention, unbiasedness of O over many offsets, and
central finite differences of the dropped loss.
"""
from __future__ import annotations

import numpy as np

# Philox-4x32 round multipliers and Weyl key increments (SC'11 paper, section 3).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds on broadcastable uint32 counter words.

    One round: the two 32x32 -> 64-bit products M0*c0 and M1*c2 are split into
    high and low halves; the new counter is (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
    hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key is then bumped by (W0, W1) mod 2^32.
    Returns the four output words as uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3))
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    sh = np.uint64(32)
    for _ in range(PHILOX_ROUNDS):
        p0 = np.uint64(PHILOX_M0) * c0       # < 2^64: exact in uint64
        p1 = np.uint64(PHILOX_M1) * c2
        c0, c1, c2, c3 = ((p1 >> sh) ^ c1 ^ k0, p1 & _MASK32, (p0 >> sh) ^ c3 ^ k1, p0 & _MASK32)
        k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
        k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def threshold(p: float) -> int:
    """Byte threshold t for drop probability p in [0, 1): round(256 p), at most 255."""
    p = float(p)
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must be in [0, 1)")
    return min(255, int(np.floor(256.0 * p + 0.5)))


def rescale(t: int) -> float:
    """1 / (1 - p') for p' = t / 256."""
    return 256.0 / (256.0 - t)


def draw_bytes(bh: int, rows, n_k: int, seed: int, offset: int) -> np.ndarray:
    """uint8 [len(rows), n_k]: the byte drawn for (query row, key) of problem bh."""
    rows = np.asarray(rows, dtype=np.int64)
    groups = (n_k + 15) // 16
    g = np.arange(groups, dtype=np.uint64)[None, :]
    i = rows.astype(np.uint64)[:, None]
    w = philox4x32_10(g, i, np.uint64(bh), np.uint64(offset), seed & 0xFFFFFFFF,
                      (seed >> 32) & 0xFFFFFFFF)
    words = np.stack(w, axis=-1)                      # [rows, groups, 4] uint32
    by = words.astype("<u4").view(np.uint8)           # little-endian bytes: word e//4, byte e%4
    return by.reshape(len(rows), groups * 16)[:, :n_k]


def keep_mask(bh: int, rows, n_k: int, seed: int, offset: int, p: float) -> np.ndarray:
    """Boolean [len(rows), n_k]: Z_ij, True where the element is kept."""
    return draw_bytes(bh, rows, n_k, seed, offset) >= threshold(p)


def multiplier(bh: int, seed: int, offset: int, p: float):
    """Function rows, n_k -> fp64 [len(rows), n_k] of Z / (1 - p'), the factor
    that turns P into the dropped probabilities of problem bh."""
    t = threshold(p)
    r = rescale(t)

    def f(rows, n_k):
        return np.where(draw_bytes(bh, rows, n_k, seed, offset) >= t, r, 0.0)

    return f
