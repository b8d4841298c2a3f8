"""Philox4x32-10 counter-based RNG and the draws the verifier consumes (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source of the generator: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11 -- the Philox-4x32 bijection
with 10 rounds.  One round maps the counter (c0, c1, c2, c3) under the key
(k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57, and the key is bumped by the Weyl
constants (0x9E3779B9, 0xBB67AE85) between rounds.

How the verifier keys it (a reading: the pages only require that randomness be
"applied consistently" -- "Speculative decoding: accelerate LLM generation
without changing its answers", section 3 -- and the method fixes Philox keyed by
seed, request, position and token):

    key     = (seed & 0xffffffff, seed >> 32)
    counter = (x >> 2, pos, request_id, stream)      output word x & 3
    stream 0: the exponential E_x of token x in the residual / bonus race
    stream 1: the accept uniform u of a draft position (token slot x = 0)

The uniform map keeps 23 random bits so that every value is exactly
representable in fp32 as well as fp64 (a 24-bit mantissa cannot hold m + 1/2
for m >= 2^23):

    U = (2 * (r >> 9) + 1) * 2^-24        in (0, 1), never 0 or 1
    E = -ln U                             Exp(1) up to the 2^-23 grid
"""

from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
ROUNDS = 10

STREAM_RACE = 0
STREAM_ACCEPT = 1

_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 of counters (c0..c3) under key (k0, k1).

    Arguments broadcast as numpy uint32 arrays (or Python ints); returns four
    uint32 arrays.  Follows the round function and key schedule of Salmon et
    al., SC'11, written with 64-bit products for the 32x32 -> 64 multiply.
    """
    c0, c1, c2, c3 = np.broadcast_arrays(
        *(np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3)))
    c0, c1, c2, c3 = (np.array(v, dtype=np.uint64) for v in (c0, c1, c2, c3))
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    for _ in range(ROUNDS):
        p0 = c0 * np.uint64(M0)          # < 2^64, exact in uint64
        p1 = c2 * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + W0) & 0xFFFFFFFF
        k1 = (k1 + W1) & 0xFFFFFFFF
    return tuple(v.astype(np.uint32) for v in (c0, c1, c2, c3))


def seed_key(seed: int):
    """Split the 64-bit verification seed into the Philox key words."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniform_from_bits(r):
    """U = (2 * (r >> 9) + 1) * 2^-24 in fp64 (exact; also exact in fp32)."""
    r = np.asarray(r, dtype=np.uint64)
    return ((r >> np.uint64(9)).astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24


def raw_words(seed, request_id, pos, stream, x):
    """The 32-bit word that keys token slot x (array) at (request, position, stream)."""
    x = np.asarray(x, dtype=np.uint64)
    k0, k1 = seed_key(seed)
    words = philox4x32_10(x >> np.uint64(2), int(pos) & 0xFFFFFFFF,
                          int(request_id) & 0xFFFFFFFF, int(stream), k0, k1)
    stacked = np.stack(words, axis=-1)            # [..., 4]
    return np.take_along_axis(stacked, (x & np.uint64(3)).astype(np.int64)[..., None],
                              axis=-1)[..., 0]


def accept_uniform(seed, request_id, pos, slot=0) -> float:
    """u for the accept test of the draft token decided at absolute position
    pos; slot = the proposal's rank among its siblings in a token tree (0 for a
    linear chain of drafts)."""
    return float(uniform_from_bits(raw_words(seed, request_id, pos, STREAM_ACCEPT,
                                             np.full(1, slot, np.uint64)))[0])


def race_exponentials(seed, request_id, pos, V) -> np.ndarray:
    """E_x = -ln U_x for every token x < V at absolute position pos (stream 0)."""
    u = uniform_from_bits(raw_words(seed, request_id, pos, STREAM_RACE,
                                    np.arange(V, dtype=np.uint64)))
    return -np.log(u)
