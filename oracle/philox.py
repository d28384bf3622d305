"""Philox4x32-10 counter-based generator, numpy, vectorised over counters.

Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
(SC'11), section 3 (the Philox S-box: two 32x32->64 multiplications per round,
the high halves XORed with the other two counter words and the round key, the
words permuted; the key advanced by the Weyl constants between rounds).  The
multipliers 0xD2511F53 / 0xCD9E8D57 and Weyl increments 0x9E3779B9 / 0xBB67AE85
are the ones the paper gives for Philox4x32.

Use in the rejection sampler ([NEURON] "Speculative Decoding (EAGLE3) in the
vLLM Neuron Framework", section "Rejection Sampling": the CPU sampler draws a
uniform per draft position for the acceptance test and exponential noise for
the Gumbel-max recovery).  Counter layout (a stated reading; the pages only say
"uniform_sample" and "exponential_noise"):

* key   = (seed mod 2^32, seed >> 32)
* counter = (block j, draft position i, request b, 2 * step_offset + purpose)
  mod 2^32 each; purpose 0 = acceptance uniform (block 0, first word),
  purpose 1 = noise for vocabulary ids 4j .. 4j+3 (word l -> id 4j + l).
* u = ((x >> 8) + 0.5) * 2^-24, exactly representable in float32; u in (0, 1).
"""
import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Apply 10 Philox4x32 rounds.  All arguments are array-likes of 32-bit values;
    returns four uint32 arrays (broadcast shape)."""
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(*(np.asarray(a, dtype=np.uint64) & _MASK
                                                   for a in (c0, c1, c2, c3, k0, k1)))
    c0, c1, c2, c3, k0, k1 = (a.copy() for a in (c0, c1, c2, c3, k0, k1))
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return tuple(a.astype(np.uint32) for a in (c0, c1, c2, c3))


def to_uniform(x):
    """32-bit word -> u = ((x >> 8) + 0.5) * 2^-24 in (0, 1), float64 (exact)."""
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(8)).astype(np.float64) + 0.5) * 2.0 ** -24


def _key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def accept_uniform(seed, step_offset, b, i):
    """Acceptance uniform of request b, draft position i."""
    k0, k1 = _key(seed)
    c3 = (2 * int(step_offset)) & 0xFFFFFFFF
    x0, _, _, _ = philox4x32_10(0, i, b, c3, k0, k1)
    return to_uniform(x0)


def noise_uniforms(seed, step_offset, b, i, V):
    """Noise uniforms for vocabulary ids 0..V-1 of request b, draft position i."""
    k0, k1 = _key(seed)
    c3 = (2 * int(step_offset) + 1) & 0xFFFFFFFF
    nblk = (V + 3) // 4
    j = np.arange(nblk, dtype=np.uint64)
    x = philox4x32_10(j, i, b, c3, k0, k1)
    words = np.stack(x, axis=-1).reshape(-1)[:V]
    return to_uniform(words)
