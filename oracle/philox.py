"""Philox4x32-10 and the acceptance uniforms (oracle side).

Philox4x32 is the counter-based generator of Salmon, Moraes, Dror and Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3" (SC'11), section 3.2: each round multiplies counter words 0 and 2
by two fixed odd 32-bit multipliers, splits the 64-bit products into high and low halves, and
mixes the high halves with counter words 1 and 3 and the round key; the round key is bumped by
two Weyl increments (the golden ratio and sqrt(3)-1, as 32-bit fractions) between rounds.  Ten
rounds are used.

The acceptance uniforms of rejection sampling ([GUIDE] section "棄却サンプリング：出力品質を保証
する") are keyed by (seed, request, node, purpose): key = (seed mod 2^32, seed >> 32), counter =
(request, node, purpose, 0); purpose 0 = accept test of a node, 1 = resample at the endpoint.
u = (2 * (x0 >> 9) + 1) * 2^-24 lies strictly inside (0, 1) and is exact in float32.
"""

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.  All arguments are broadcastable uint32-valued arrays.

    Returns the four output words as uint64 arrays holding 32-bit values.
    """
    x0, x1, x2, x3, kk0, kk1 = (np.asarray(v, dtype=np.uint64) & _MASK
                                 for v in (c0, c1, c2, c3, k0, k1))
    x0, x1, x2, x3, kk0, kk1 = np.broadcast_arrays(x0, x1, x2, x3, kk0, kk1)
    for rnd in range(10):
        if rnd:
            kk0 = (kk0 + _W0) & _MASK
            kk1 = (kk1 + _W1) & _MASK
        p0 = _M0 * x0
        p1 = _M1 * x2
        hi0, lo0 = p0 >> _S32, p0 & _MASK
        hi1, lo1 = p1 >> _S32, p1 & _MASK
        x0, x1, x2, x3 = hi1 ^ x1 ^ kk0, lo1, hi0 ^ x3 ^ kk1, lo0
    return x0, x1, x2, x3


def uniforms(seed, request, node, purpose):
    """Acceptance uniforms u(seed, request, node, purpose) in (0, 1) as float64 (exact)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    x0, _, _, _ = philox4x32_10(request, node, purpose, 0, seed & 0xFFFFFFFF, seed >> 32)
    return ((x0 >> np.uint64(9)).astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24
