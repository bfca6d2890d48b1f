"""Philox4x32-10 and the sampler's uniform stream (test oracle).

Philox is written from its published definition (J. K. Salmon, M. A. Moraes,
R. O. Dror, D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
SC'11, section on the Philox family): a 4x32-bit counter and a 2x32-bit key;
each of 10 rounds multiplies counter words 0 and 2 by two fixed 32-bit
multipliers, takes the high and low halves of the 64-bit products, and
xors the high halves with the other counter words and the round key; the
key is bumped by two Weyl constants between rounds.

Stream used by the sampler (one written specification, implemented twice,
here and in the CUDA kernel):
    key     = (lo32(seed), hi32(seed))
    counter = (j // 4, lo32(offset), hi32(offset), 0)
    w_j     = word (j % 4) of Philox4x32-10(counter, key)
    u_j     = ((w_j >> 9) + 0.5) * 2**-23        in (0, 1)
so one Philox evaluation feeds four consecutive vocabulary ids.  The 23-bit
grid keeps u_j exactly representable in float32 (m + 1/2 with m < 2**23 has
24 significant bits), so both implementations start from the same u_j.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def _mulhilo(a: np.ndarray, m: int):
    prod = a.astype(np.uint64) * np.uint64(m)
    return (prod >> np.uint64(32)).astype(np.uint64), (prod & np.uint64(MASK32)).astype(np.uint64)


def philox4x32_10(counter, key):
    """Vectorised Philox4x32-10.

    counter: sequence of 4 arrays (or ints) of uint32 words; key: 2 words.
    Returns four uint32 arrays.
    """
    c = [np.asarray(x, dtype=np.uint64) & np.uint64(MASK32) for x in counter]
    c = list(np.broadcast_arrays(*c))
    k0 = np.uint64(int(key[0]) & MASK32)
    k1 = np.uint64(int(key[1]) & MASK32)
    for rnd in range(10):
        hi0, lo0 = _mulhilo(c[0], PHILOX_M0)
        hi1, lo1 = _mulhilo(c[2], PHILOX_M1)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        if rnd != 9:
            k0 = np.uint64((int(k0) + PHILOX_W0) & MASK32)
            k1 = np.uint64((int(k1) + PHILOX_W1) & MASK32)
    return [x.astype(np.uint32) for x in c]


def stream_words(seed: int, offset: int, ids: np.ndarray) -> np.ndarray:
    """Word w_j of the sampler stream for each vocabulary id in ``ids``."""
    ids = np.asarray(ids, dtype=np.uint64)
    seed, offset = int(seed), int(offset)
    key = (seed & MASK32, (seed >> 32) & MASK32)
    ctr = (ids >> np.uint64(2), np.uint64(offset & MASK32),
           np.uint64((offset >> 32) & MASK32), np.uint64(0))
    words = philox4x32_10(ctr, key)
    lane = (ids & np.uint64(3)).astype(np.int64)
    stacked = np.stack([np.broadcast_to(w, ids.shape) for w in words], axis=0)
    return stacked[lane, np.arange(ids.shape[0])] if ids.ndim == 1 else stacked


def uniforms(seed: int, offset: int, ids: np.ndarray) -> np.ndarray:
    """u_j = ((w_j >> 9) + 0.5) * 2**-23 as float64 (exact in float32 too)."""
    w = stream_words(seed, offset, ids).astype(np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(seed: int, offset: int, ids: np.ndarray) -> np.ndarray:
    """g_j = -log(-log(u_j)) in float64."""
    return -np.log(-np.log(uniforms(seed, offset, ids)))
