"""Exact gradients of scaled-dot-product attention in float64 -- test infrastructure.

Only tests/, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline use
this module; the CUDA path never imports it and shares no code with it.

What is computed is the plain definition: the chain rule through
O = P V, P = softmax(S) row by row, S = scale * Q K^T (+ mask), written out.
The page "4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization &
FP8", section "The backward pass: recompute, and the one identity that makes
it tile-able", lists the same quantities for one head, given the incoming
gradient dO:
  dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),   dQ = scale * dS K,
  dK = scale * dS^T Q,
with D_i = sum_j P_ij dP_ij -- the softmax Jacobian applied to a row of dP.
(The page then rewrites D_i as the row dot product of dO_i and O_i; that
identity is what a tiled kernel uses, and the tests pin it separately.  The
page recovers P from the saved logsumexp; here P is the softmax itself.)
Masks are the forward's: causal top-left (key j visible from query i iff
j <= i) and, with a window w, also j > i - w ("4.3", Exercise 5).  A row with
no visible key has P = 0.  With grouped KV heads (query head h reads KV head
h // (H / H_kv), "4.3", section "Calling the real kernel"), the chain rule sums
the contributions of every query head that reads a KV head into its dK, dV.
"""
from __future__ import annotations

import numpy as np


def softmax_weights(q, k, scale: float, causal: bool, window: int = 0):
    """P [N, N] of one (batch, head): masked, row-normalised exp of the scores."""
    N = k.shape[0]
    S = scale * (q @ k.T)
    if causal:
        i = np.arange(N)[:, None]
        j = np.arange(N)[None, :]
        vis = j <= i
        if window > 0:
            vis &= j > i - window
        S = np.where(vis, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    live = np.isfinite(m)
    E = np.where(np.isfinite(S), np.exp(S - np.where(live, m, 0.0)), 0.0)
    ell = E.sum(axis=1, keepdims=True)
    return np.where(live, E / np.where(live, ell, 1.0), 0.0)


def backward_head(q, k, v, dO, scale: float, causal: bool, window: int = 0):
    """(dQ, dK, dV) of one (batch, head); all arrays [N, d] float64."""
    P = softmax_weights(q, k, scale, causal, window)
    dV = P.T @ dO
    dP = dO @ v.T
    D = (P * dP).sum(axis=1)              # Jacobian of the row softmax applied to dP
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV


def backward(q, k, v, dO, scale: float, causal: bool, window: int = 0):
    """Gradients for [B, H, N, d] q, dO and [B, H_kv, N, d] k, v (H_kv | H).
    Returns (dQ [B, H, N, d], dK [B, H_kv, N, d], dV [B, H_kv, N, d])."""
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if H % H_kv:
        raise ValueError("KV heads must divide query heads")
    group = H // H_kv
    dQ = np.zeros_like(q, dtype=np.float64)
    dK = np.zeros(k.shape, dtype=np.float64)
    dV = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = h // group
            a, bk, c = backward_head(q[b, h], k[b, g], v[b, g], dO[b, h], scale, causal, window)
            dQ[b, h] = a
            dK[b, g] += bk
            dV[b, g] += c
    return dQ, dK, dV


def row_dot(dO, O):
    """D_i = sum_t dO_it O_it: the page's form of D (used by the tests only)."""
    return (dO * O).sum(axis=-1)


def backward_sampled(q, k, v, dO, scale: float, causal: bool, rows, keys, window: int = 0):
    """The same definition restricted to some outputs of one (batch, head):
    dQ for the listed query ``rows`` and dK, dV for the listed ``keys``.

    Row i of dQ needs row i of P and dP; key j of dK, dV needs column j of P,
    which needs every row's normaliser: the softmax is taken row by row over
    all keys (in chunks of rows, so that no N x N array is formed)."""
    N = k.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)

    def prob_rows(r):
        S = scale * (q[r] @ k.T)
        if causal:
            j = np.arange(N)[None, :]
            vis = j <= r[:, None]
            if window > 0:
                vis &= j > r[:, None] - window
            S = np.where(vis, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        live = np.isfinite(m)
        E = np.where(np.isfinite(S), np.exp(S - np.where(live, m, 0.0)), 0.0)
        ell = E.sum(axis=1, keepdims=True)
        return np.where(live, E / np.where(live, ell, 1.0), 0.0)

    # dQ rows: full rows of P and dP.
    P = prob_rows(rows)
    dP = dO[rows] @ v.T
    D = (P * dP).sum(axis=1)
    dQ = scale * ((P * (dP - D[:, None])) @ k)
    # dK, dV keys: the listed columns of P for all rows, plus every row's D.
    dK = np.zeros((keys.size, q.shape[1]))
    dV = np.zeros((keys.size, v.shape[1]))
    for c0 in range(0, N, 512):
        r = np.arange(c0, min(N, c0 + 512))
        Pr = prob_rows(r)
        dPr = dO[r] @ v.T
        Dr = (Pr * dPr).sum(axis=1)
        Pc = Pr[:, keys]
        dSc = Pc * (dPr[:, keys] - Dr[:, None])
        dV += Pc.T @ dO[r]
        dK += scale * (dSc.T @ q[r])
    return dQ, dK, dV
