"""q8_0 block quantisation and the f16 cache rounding, written out from the definition.

Source: the pages run with a "q8_0 device-resident cache" (llama.cpp PR #58,
"completion : allow the prompt to be processed under its own split mode",
section "Why") and an "f16 cache" (llama.cpp PR #59, "llama : switch the split
mode of a live context", section "Why"), without defining either.  The reading
taken here is the standard q8_0 block: 32 consecutive values along head_dim
share one fp16 scale d = amax/127 and are stored as int8 codes q = round(x/d).

All arithmetic is IEEE float32 in this order (the order a kernel can repeat
bit for bit):
    amax = max_i |x_i|                 exact
    d    = amax / 127                  float32 division, correctly rounded
    q_i  = round(x_i / d)              float32 division, then round half away
                                       from zero; all codes 0 when d == 0
                                       (amax == 0, or amax so small that
                                       amax/127 underflows: x/d is undefined)
    d_h  = fp16(d)                     round to nearest even, subnormals kept
Dequantisation: xhat_i = float(d_h) * q_i, exact in float32 (11 x 8 bits).
The f16 cache stores fp16(x) with round to nearest even.
"""

import numpy as np

BLOCK = 32


def quantize_blocks(x):
    """Quantise float32 values [..., n] (n a multiple of 32) into q8_0 blocks.

    Returns (d_h, q): d_h float16 [..., n/32] (the block scales), q int8 [..., n].
    """
    x = np.asarray(x, dtype=np.float32)
    if not np.isfinite(x).all():
        raise ValueError("q8_0 quantisation is defined for finite inputs only")
    shape = x.shape
    if shape[-1] % BLOCK:
        raise ValueError("last axis must be a multiple of 32")
    xb = x.reshape(shape[:-1] + (shape[-1] // BLOCK, BLOCK))
    amax = np.abs(xb).max(axis=-1)
    d = amax / np.float32(127.0)                      # float32 / float32 -> float32
    nonzero = d > 0
    divisor = np.where(nonzero, d, np.float32(1.0)).astype(np.float32)
    ratio = xb / divisor[..., None]                   # float32 division, correctly rounded
    r = ratio.astype(np.float64)                      # exact widening; |r| + 0.5 is exact too
    q = np.sign(r) * np.floor(np.abs(r) + 0.5)        # round half away from zero
    q = np.where(nonzero[..., None], q, 0.0)
    q = np.clip(q, -127, 127).astype(np.int8).reshape(shape)
    d_h = d.astype(np.float16)                        # round to nearest even
    return d_h, q


def dequantize_blocks(d_h, q):
    """float32 values d_h * q for q8_0 blocks (d_h [..., n/32] float16, q [..., n] int8)."""
    q = np.asarray(q)
    shape = q.shape
    qb = q.reshape(shape[:-1] + (shape[-1] // BLOCK, BLOCK)).astype(np.float32)
    return (np.asarray(d_h).astype(np.float32)[..., None] * qb).reshape(shape)


def to_f16(x):
    """The f16 cache value of float32 inputs: fp16 with round to nearest even."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)
