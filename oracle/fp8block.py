"""Blockwise FP8 quantise-dequantise, CPU oracle (TEST INFRASTRUCTURE ONLY).

The pages list blockwise FP8 as the Hopper precision of the fused kernel ("How does
the fused kernel work?": BF16, MXFP8 on Blackwell, blockwise FP8 on Hopper) without
its details.  Reading, in the form Blackwell tensor cores take (power-of-two scales):
  * activations: blocks of 128 consecutive elements along the GEMM's contraction axis
    (one token's 128 channels; along the token axis for the weight-gradient
    operands, 128 rows from the expert's first, the tail zero-padded);
  * weights: 128 x 128 blocks of the [rows, cols] matrix (one scale per block, the
    same blocks whichever axis a GEMM contracts);
  * scale X = 2 ** ceil(log2(amax / 448)), the smallest power of two that keeps every
    element of the block within E4M3's +-448 (X = 2 ** -127 for an all-zero block,
    exponents clipped to [-127, 127]);
  * each element is v / X rounded to nearest-even E4M3 and dequantised as e4m3 * X.
"""
from __future__ import annotations

import numpy as np

from .mx import e4m3_round

BLOCK = 128
E4M3_MAX = 448.0


def ue8m0_ceil_exponent(amax: np.ndarray) -> np.ndarray:
    """ceil(log2(amax / 448)), clipped to [-127, 127]; -127 for amax = 0 (int)."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E4M3_MAX))
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def _qdq_blocks(blocks: np.ndarray, amax: np.ndarray) -> np.ndarray:
    scale = np.exp2(ue8m0_ceil_exponent(amax).astype(np.float64))
    return e4m3_round(blocks / scale) * scale


def qdq_1d(v: np.ndarray, axis: int, block: int = BLOCK) -> np.ndarray:
    """Blocks of `block` consecutive elements along `axis` (a trailing partial block
    counts as zero-padded)."""
    v = np.asarray(v, dtype=np.float64)
    moved = np.moveaxis(v, axis, -1)
    n = moved.shape[-1]
    nb = -(-n // block) if n else 0
    pad = nb * block - n
    if pad:
        moved = np.concatenate([moved, np.zeros(moved.shape[:-1] + (pad,))], axis=-1)
    blocks = moved.reshape(moved.shape[:-1] + (nb, block))
    amax = np.abs(blocks).max(axis=-1, keepdims=True, initial=0.0)
    deq = _qdq_blocks(blocks, amax).reshape(moved.shape)[..., :n]
    return np.moveaxis(deq, -1, axis)


def qdq_2d(W: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """block x block tiles of the last two axes (their sizes multiples of block)."""
    W = np.asarray(W, dtype=np.float64)
    r, c = W.shape[-2:]
    if r % block or c % block:
        raise ValueError("weight dimensions must be multiples of the block")
    t = W.reshape(W.shape[:-2] + (r // block, block, c // block, block))
    amax = np.abs(t).max(axis=(-3, -1), keepdims=True)
    return _qdq_blocks(t, amax).reshape(W.shape)
