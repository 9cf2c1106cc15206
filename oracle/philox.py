"""Philox4x32-10 counter-based generator and the uniforms the SMC-SD step draws.

Test infrastructure: part of the CPU oracle (see ``oracle/__init__.py``).

The pages fix that each random choice of the step (bonus token, SpS acceptance,
SpS residual token, systematic-resampling offset) is a uniform draw; they do not
name a generator.  The oracle and the CUDA path each implement Philox4x32-10
from its published definition (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11): a 4x32-bit counter, a 2x32-bit key, ten
rounds of two 32x32->64 multiplies, with the key bumped by the Weyl constants
between rounds.

Keying used by both sides (a reading of the pages, which are silent here):
    key     = (seed mod 2^32, seed >> 32)
    counter = (step, stream, position, purpose)
where ``stream`` is the global particle index b*N+n for the bonus token and the
prompt index b for the other purposes.  The uniform is built from output word 0
as (x0 >> 8) * 2^-24, which is exact in both fp32 and fp64, so both sides
compare the same number.
"""
import numpy as np

MASK32 = 0xFFFFFFFF

# Round multipliers and key increments of Philox4x32 (published definition).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85

# Purposes (4th counter word).
DRAFT = 0       # reserved for the extend-side draft sampler
BONUS = 1       # bonus token of a particle, position K
ACCEPT = 2      # SpS acceptance test of drafted position k
RESIDUAL = 3    # SpS residual token after the first rejection at position j
RESAMPLE = 4    # systematic-resampling offset u0 of a prompt, position 0


def philox4x32_10(counter, key):
    """One Philox4x32-10 block: 4 counter words and 2 key words -> 4 words.

    Scalar pure-Python version, written round by round from the definition.
    """
    c0, c1, c2, c3 = (int(w) & MASK32 for w in counter)
    k0, k1 = (int(w) & MASK32 for w in key)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> 32, p0 & MASK32
        hi1, lo1 = p1 >> 32, p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 over numpy arrays of counter/key words.

    Same rounds as ``philox4x32_10``; products are formed in uint64 so the
    high and low halves are exact.  Used for the large empirical-histogram
    pins, where a Python loop per draw would be too slow.
    """
    arrs = np.broadcast_arrays(*(np.asarray(w, dtype=np.uint64) & np.uint64(MASK32)
                                 for w in (c0, c1, c2, c3, k0, k1)))
    c0, c1, c2, c3, k0, k1 = (a.copy() for a in arrs)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    w0, w1 = np.uint64(PHILOX_W0), np.uint64(PHILOX_W1)
    mask = np.uint64(MASK32)
    sh = np.uint64(32)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + w0) & mask
            k1 = (k1 + w1) & mask
        p0 = m0 * c0
        p1 = m1 * c2
        hi0, lo0 = p0 >> sh, p0 & mask
        hi1, lo1 = p1 >> sh, p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform(seed, step, stream, position, purpose):
    """u in [0, 1) on the 2^-24 lattice for one (seed, step, stream, position, purpose)."""
    seed = int(seed)
    x0 = philox4x32_10((step, stream, position, purpose),
                       (seed & MASK32, (seed >> 32) & MASK32))[0]
    return (x0 >> 8) * 2.0 ** -24


def uniform_np(seed, step, stream, position, purpose):
    """Vectorised ``uniform``: any argument may be an integer array."""
    seed = np.asarray(seed, dtype=np.uint64)
    x0 = philox4x32_10_np(step, stream, position, purpose,
                          seed & np.uint64(MASK32), seed >> np.uint64(32))[0]
    return (x0 >> np.uint64(8)).astype(np.float64) * 2.0 ** -24
