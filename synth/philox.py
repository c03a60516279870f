"""Philox4x32-10 counter-based generator and the sampler's uniform draws.

Philox4x32-10 is defined in Salmon, Moraes, Dror and Shaw, "Parallel random
numbers: as easy as 1, 2, 3" (SC'11): a 4-word counter is passed through ten
rounds of two 32x32->64-bit multiplies, each round mixing in the 2-word key,
which is advanced by the Weyl constants between rounds.

The decode workloads draw one uniform number per sampled token from a seeded
Philox stream.  The draw for (step, row, stream) takes the first output word
``w`` of counter ``(step, row, stream, 0)`` under key ``(seed, 0)`` and maps it
to ``u = (w >> 8) * 2**-24`` in [0, 1).  ``stream`` is 0 for the T3 / Talker
sampler and j for code-predictor pass j.  The draws are inputs of the decode
step (passed to both implementations), never regenerated inside either one.
"""

from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter: np.ndarray, key: tuple[int, int]) -> np.ndarray:
    """Apply Philox4x32-10 to an array of counters.

    counter: uint32 array of shape [..., 4]; key: two 32-bit words.
    Returns a uint32 array of the same shape.
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniform_draws(seed: int, n_steps: int, n_rows: int, n_streams: int = 1,
                  step0: int = 0) -> np.ndarray:
    """Uniform draws u[step][row][stream] in [0, 1) as float32 (24-bit grid).

    Each value is exactly representable in fp32, so both implementations see
    the same number.
    """
    s, r, t = np.meshgrid(np.arange(step0, step0 + n_steps), np.arange(n_rows),
                          np.arange(n_streams), indexing="ij")
    ctr = np.stack([s, r, t, np.zeros_like(s)], axis=-1).astype(np.uint32)
    w = philox4x32_10(ctr, (seed, 0))[..., 0]
    return ((w >> 8).astype(np.float64) * 2.0 ** -24).astype(np.float32)
