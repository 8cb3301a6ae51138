"""Sylvester Hadamard matrix and fast Walsh-Hadamard transform -- test infrastructure.

Source: "4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization &
FP8", section "Incoherent processing: rotate away the outliers": the Sylvester
construction doubles [[H, H], [H, -H]] from the 1x1 matrix [1] and divides by
sqrt(n) so the result is orthonormal; the rotation is M = H D with D a random
diagonal of +-1, applied as x M to rows x of Q and K, and the page notes that
it can be applied in O(d log d) with the fast Hadamard transform.
"""
from __future__ import annotations

import numpy as np


def sylvester(n: int) -> np.ndarray:
    """Orthonormal n x n Sylvester Hadamard matrix (n a power of two), float64."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H / np.sqrt(n)


def fwht(x: np.ndarray) -> np.ndarray:
    """x @ sylvester(n) along the last axis, by butterflies (float64).

    Stage with half-width h pairs elements i and i + h inside each block of
    2h and replaces them with (a + b, a - b); after log2(n) stages the result
    is divided by sqrt(n).
    """
    y = np.array(x, dtype=np.float64, copy=True)
    n = y.shape[-1]
    if n & (n - 1):
        raise ValueError("last axis must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < n:
        y = y.reshape(*lead, n // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(*lead, n)
        h *= 2
    return y / np.sqrt(n)


def rotation(signs: np.ndarray) -> np.ndarray:
    """The orthogonal matrix M = H diag(signs) for one head (float64)."""
    signs = np.asarray(signs, dtype=np.float64)
    return sylvester(signs.size) * signs[None, :]
