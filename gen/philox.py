"""Philox4x32-10 counter-based generator (input generation only).

Written from the published definition of Philox (Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): a 4x32-bit
counter and a 2x32-bit key go through ten rounds; each round multiplies two
counter words by fixed odd constants, keeps the 64-bit products' high and
low halves, and mixes the high halves with the other two counter words and
the round key; the key is advanced by two Weyl constants between rounds.

The verification walk of tree speculative sampling consumes uniform random
numbers.  They are drawn here, once, and handed to both the CUDA path and the
oracle as an ordinary input tensor, so neither side implements a generator.
"""
import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)
_SHIFT32 = np.uint64(32)


def philox4x32_10(counter, key):
    """Apply Philox4x32-10 to a batch of counters.

    counter: uint32-valued array of shape [..., 4]; key: two uint32 values
    (or an array broadcastable to [..., 2]).  Returns uint32 array [..., 4].
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK32
    k = np.broadcast_to(np.asarray(key, dtype=np.uint64) & _MASK32,
                        c.shape[:-1] + (2,)).copy()
    x0, x1, x2, x3 = (c[..., i].copy() for i in range(4))
    k0, k1 = k[..., 0], k[..., 1]
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _W0) & _MASK32
            k1 = (k1 + _W1) & _MASK32
        p0 = _M0 * x0          # < 2**64: both factors are 32-bit
        p1 = _M1 * x2
        hi0, lo0 = p0 >> _SHIFT32, p0 & _MASK32
        hi1, lo1 = p1 >> _SHIFT32, p1 & _MASK32
        x0, x1, x2, x3 = (hi1 ^ x1 ^ k0), lo1, (hi0 ^ x3 ^ k1), lo0
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def uint32_to_unit_float(words):
    """Map uint32 words to float32 uniforms in [0, 1): (w >> 8) * 2**-24.

    The top 24 bits are kept, so every value is exactly representable in
    float32 and the map never returns 1.0.
    """
    w = np.asarray(words, dtype=np.uint32) >> np.uint32(8)
    return (w.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def tree_uniforms(seed, batch, n_nodes):
    """Uniforms u[b, i, 0:2] for the verification walk, float32 [B, n, 2].

    Counter (b, i, 0, 0), key (seed low 32 bits, seed high 32 bits); words 0
    and 1 of the output block become u[b, i, 0] (accept test of node i) and
    u[b, i, 1] (bonus draw at node i).
    """
    b = np.arange(batch, dtype=np.uint64)[:, None]
    i = np.arange(n_nodes, dtype=np.uint64)[None, :]
    ctr = np.zeros((batch, n_nodes, 4), dtype=np.uint64)
    ctr[..., 0] = b
    ctr[..., 1] = i
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)
    out = philox4x32_10(ctr, key)
    return uint32_to_unit_float(out[..., :2])
