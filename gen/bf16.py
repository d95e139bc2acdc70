"""bfloat16 storage helpers for NumPy (which has no bfloat16 type).

bf16 tensors are carried as ``uint16`` bit patterns.  Rounding from float32 is round to nearest,
ties to even, which is what ``torch.Tensor.to(torch.bfloat16)`` does for finite values.
"""

import numpy as np

_CHUNK = 1 << 24


def f32_to_bf16_bits(x):
    """Round a float32 array to bf16 and return the bit patterns as uint16 (same shape)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    xf = x.reshape(-1)
    of = out.reshape(-1)
    for s in range(0, xf.size, _CHUNK):
        u = xf[s:s + _CHUNK].view(np.uint32)
        # finite inputs never carry into the sign bit: the largest finite magnitude is 0x7F7FFFFF
        r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
        of[s:s + _CHUNK] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(b):
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b):
    """Exact widening of bf16 bit patterns to float64."""
    return bf16_bits_to_f32(b).astype(np.float64)


def normal_bf16(rng, shape, std=1.0):
    """Draw N(0, std^2) in float32 chunk by chunk and store the bf16-rounded bits."""
    out = np.empty(shape, dtype=np.uint16)
    of = out.reshape(-1)
    for s in range(0, of.size, _CHUNK):
        n = min(_CHUNK, of.size - s)
        v = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        of[s:s + n] = f32_to_bf16_bits(v)
    return out
