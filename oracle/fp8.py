"""Incoherent processing and block FP8 quantisation of Q, K, V -- test infrastructure.

Sources:
  * "4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization & FP8",
    section "Incoherent processing: rotate away the outliers": Q and K are
    multiplied by the same orthogonal M = H D (H orthonormal Sylvester, D a
    random +-1 diagonal) before quantisation, so (QM)(KM)^T = QK^T; a scale
    s = amax / 448 brings values into the E4M3 range (s = 1 when amax = 0).
    Section "What stays in higher precision": operands are FP8, accumulation
    and the softmax statistics are not.
  * "FlashAttention-3: How Warp Specialization, Asynchronous TMA Tiling, and
    FP8 Hardware Acceleration Scale Attention on Hopper GPUs", section 4: one
    scaling factor per block of each of Q, K, V; a score tile is
    s_Q * s_K * (Q8 K8^T).

Readings where the pages leave a step open: the block is 128 consecutive rows
of one (batch, head) over all d columns; V is quantised per block but not
rotated (the rotation is needed only where the two operands meet in a dot
product, Q with K); the signs are one draw per head shared by Q and K.
"""
from __future__ import annotations

import numpy as np

from . import e4m3, hadamard

BLOCK_ROWS = 128


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x M per head: x [B, H, N, d] float64, signs [H, d] of +-1 -> float64."""
    y = hadamard.fwht(x)
    return y * np.asarray(signs, dtype=np.float64)[None, :, None, :]


def block_amax(x: np.ndarray, block: int = BLOCK_ROWS) -> np.ndarray:
    """max |x| over each block of ``block`` rows (all d columns): [B, H, nblk]."""
    B, H, N, d = x.shape
    nb = -(-N // block)
    pad = nb * block - N
    a = np.abs(x)
    if pad:
        a = np.concatenate([a, np.zeros((B, H, pad, d))], axis=2)
    return a.reshape(B, H, nb, block * d).max(axis=-1)


def block_scales(x: np.ndarray, block: int = BLOCK_ROWS) -> np.ndarray:
    """s = amax / 448 per block, or 1 where the block is all zero."""
    amax = block_amax(x, block)
    return np.where(amax > 0, amax / e4m3.MAX_FINITE, 1.0)


def quantize(x: np.ndarray, scales: np.ndarray, block: int = BLOCK_ROWS) -> np.ndarray:
    """E4M3 codes of x / s with s the scale of each row's block: uint8 [B, H, N, d]."""
    N = x.shape[2]
    s_rows = np.repeat(scales, block, axis=2)[:, :, :N, None]
    return e4m3.encode(x / s_rows)


def dequantize(codes: np.ndarray, scales: np.ndarray, block: int = BLOCK_ROWS) -> np.ndarray:
    """codes * s, float64 [B, H, N, d]."""
    N = codes.shape[2]
    s_rows = np.repeat(scales, block, axis=2)[:, :, :N, None]
    return e4m3.decode(codes) * s_rows


def prepare(q, k, v, signs, block: int = BLOCK_ROWS):
    """Full preparation of the FP8 operands from float64 inputs.

    Returns a dict with the rotated float64 q', k' and, for each of q, k, v,
    the E4M3 codes [B, H, N, d] (V in its natural row layout) and the block
    scales [B, H, nblk].
    """
    qr = rotate(q, signs)
    kr = rotate(k, signs)
    out = {"q_rot": qr, "k_rot": kr}
    for name, x in (("q", qr), ("k", kr), ("v", np.asarray(v, dtype=np.float64))):
        s = block_scales(x, block)
        out[name + "_scale"] = s
        out[name + "8"] = quantize(x, s, block)
    return out
