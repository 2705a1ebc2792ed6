"""MXFP8 block quantise-dequantise, CPU oracle (TEST INFRASTRUCTURE ONLY).

The pages name MXFP8 as the Blackwell precision of the fused kernel
("How does the fused kernel work?": BF16, MXFP8 Blackwell only, blockwise FP8
Hopper only) without its details.  The reading used here is the OCP
Microscaling (MX) v1.0 format for MXFP8:
  * a block is 32 consecutive elements along the contraction (K) axis;
  * the shared scale is a power of two stored as E8M0:
        X = 2 ** (floor(log2(amax)) - 8)          (8 = largest exponent of E4M3)
    and X = 2 ** -127 (every element 0) for an all-zero block;
  * each element is v / X rounded to nearest-even E4M3 (the 'fn' variant: no
    infinities, largest finite 448, smallest subnormal 2**-9), saturating at
    +-448, and dequantised as e4m3 * X.
bf16_round gives the bfloat16 value of a number: the layer stores its
intermediates in bf16, and in the MXFP8 modes an element's e4m3 rounding is
decided on that stored value.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8            # exponent of the largest normal E4M3 value (448 = 1.75 * 2**8)
E4M3_EMIN = -6           # smallest normal exponent
E4M3_MBITS = 3
E8M0_MIN_EXP = -127
E8M0_MAX_EXP = 127


def e4m3_round(q: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_EMIN)                       # subnormals share the 2**-6 binade step
    step = np.exp2(e - E4M3_MBITS)
    r = np.rint(a / step) * step                        # numpy rint: round half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, q)


BF16_MBITS = 7           # stored fraction bits of bfloat16
BF16_EMIN = -126         # smallest normal exponent (that of fp32)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even): 8 significant bits and
    fp32's exponent range, subnormals in steps of 2**-133.  Finite inputs below
    the bf16 overflow threshold only."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.exp2(np.maximum(e, BF16_EMIN) - BF16_MBITS)
    return np.copysign(np.rint(a / step) * step, v)


def e8m0_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared-scale exponent of a block with absolute maximum `amax` (int)."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - E4M3_EMAX
    e = np.where(amax > 0, e, E8M0_MIN_EXP)
    return np.clip(e, E8M0_MIN_EXP, E8M0_MAX_EXP).astype(np.int64)


def mx_qdq(v: np.ndarray, axis: int) -> np.ndarray:
    """Quantise `v` to MXFP8 in blocks of 32 along `axis` and return the dequantised
    values.  A trailing partial block is treated as zero-padded to 32."""
    v = np.asarray(v, dtype=np.float64)
    moved = np.moveaxis(v, axis, -1)
    n = moved.shape[-1]
    nb = -(-n // BLOCK) if n else 0
    pad = nb * BLOCK - n
    if pad:
        moved = np.concatenate([moved, np.zeros(moved.shape[:-1] + (pad,))], axis=-1)
    blocks = moved.reshape(moved.shape[:-1] + (nb, BLOCK))
    amax = np.abs(blocks).max(axis=-1, initial=0.0)
    scale = np.exp2(e8m0_scale_exponent(amax).astype(np.float64))[..., None]
    deq = e4m3_round(blocks / scale) * scale
    deq = deq.reshape(moved.shape)[..., :n]
    return np.moveaxis(deq, -1, axis)
