"""Exact scaled-dot-product attention in float64 -- test infrastructure.

Sources (page titles, with the part of each page that is followed):
  * "Learn: The Memory Wall & FlashAttention", section 5.1 "Deriving the
    online softmax": safe softmax with the row max subtracted; the streaming
    state (m, l, o) initialised to (-inf, 0, 0) and updated per key block with
    the rescale factor alpha = exp(m_old - m_new); one final division o / l.
    Section 5.3 defines the logsumexp L = m + log(l); section 10, practice
    problem 2, is a worked example with printed numbers (pinned in the tests).
  * "Flash Attention series" (l1cachedell.github.io), section 2.2 "Online
    Softmax": safe softmax done in three passes -- the row max, then the sum
    of exponentials, then the division.
  * "4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization & FP8",
    section "Edit 1 -- defer the rescaling": causal masking is top-left
    aligned, key j is visible from query i iff j <= i.
  * "FlashAttention-3 & GPU Kernel Optimization: Accelerating Transformer
    Attention", section "Online softmax tiling mathematics": the merge of two
    partial softmax states (m1, l1, O1) and (m2, l2, O2).
  * "4.3 FlashAttention 2 & 3", section "Calling the real kernel": grouped-query
    attention, where KV heads divide the query heads and query head h reads KV
    head h // (H / H_kv); Exercise 5: a causal sliding window of width w, query
    i sees keys j with i - w < j <= i.

Conventions: q, k, v are float64 arrays [B, H, N, d]; ``scale`` multiplies the
raw dot products; lse is the natural log of the sum of exp of the *scaled*
scores, so that P_ij = exp(S_ij - lse_i).  A row with no visible key has
O = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np


def three_pass_rows(q, k, v, scale: float, causal: bool, rows, window: int = 0):
    """Three-pass attention for the listed query rows of one (batch, head).

    q: [N, d], k: [N, d], v: [N, d] float64.  Returns (O [len(rows), d],
    lse [len(rows)]).  The score row S_i is materialised in full.  window > 0
    (causal only) additionally hides keys j <= i - window.
    """
    rows = np.asarray(rows, dtype=np.int64)
    N = k.shape[0]
    out = np.zeros((rows.size, v.shape[1]), dtype=np.float64)
    lse = np.full(rows.size, -np.inf, dtype=np.float64)
    if rows.size == 0:
        return out, lse
    # Scores for all listed rows against all keys (one library matmul).
    S = scale * (q[rows] @ k.T)
    if causal:
        keys = np.arange(N)[None, :]
        S = np.where(keys <= rows[:, None], S, -np.inf)
        if window > 0:
            S = np.where(keys > rows[:, None] - window, S, -np.inf)
    # Pass 1: row max over visible keys.
    m = S.max(axis=1)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    # Pass 2: sum of exponentials referenced to the row max.
    E = np.exp(S - m_safe[:, None])
    E = np.where(np.isfinite(S), E, 0.0)
    ell = E.sum(axis=1)
    # Pass 3: normalised weights times V.
    with np.errstate(invalid="ignore", divide="ignore"):
        P = E / np.where(live, ell, 1.0)[:, None]
    out[live] = P[live] @ v
    lse[live] = m[live] + np.log(ell[live])
    return out, lse


def attention(q, k, v, scale: float, causal: bool, rows=None, row_chunk: int = 512,
              window: int = 0):
    """Three-pass attention for every (batch, head).

    q: [B, H, N, d]; k, v: [B, H_kv, N, d] with H_kv dividing H (query head h
    reads KV head h // (H / H_kv)).  If ``rows`` is given, only those query rows
    are computed (the same rows for every (b, h)); outputs then have N replaced
    by len(rows).  window > 0 with causal: sliding window of that many keys.
    Returns (O, lse) as float64 arrays.
    """
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if H % H_kv:
        raise ValueError("KV heads must divide query heads")
    group = H // H_kv
    sel = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((B, H, sel.size, v.shape[-1]), dtype=np.float64)
    L = np.zeros((B, H, sel.size), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for c0 in range(0, sel.size, row_chunk):
                r = sel[c0:c0 + row_chunk]
                o, l = three_pass_rows(q[b, h], k[b, h // group], v[b, h // group], scale,
                                       causal, r, window)
                O[b, h, c0:c0 + r.size] = o
                L[b, h, c0:c0 + r.size] = l
    return O, L


def probabilities(q, k, scale: float, causal: bool):
    """The full softmax weight matrix P [N, N] of one (batch, head) (tiny inputs)."""
    N = k.shape[0]
    S = scale * (q @ k.T)
    if causal:
        S = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None], S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    return E / E.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# Streaming forms, used only by the tests to pin ``three_pass_rows``.
# ---------------------------------------------------------------------------

def _rescale(alpha, acc):
    """Re-reference an accumulator to a new running max: multiply by alpha."""
    return alpha * acc


def online_row(s, vals, block: int):
    """Online-softmax recurrence over one score row, ``block`` keys at a time.

    s: [n] scaled scores (already masked, -inf where invisible), vals: [n, dv].
    Follows the state update of section 5.1: per block t with local max
    m~(t), m(t) = max(m(t-1), m~(t)), alpha(t) = exp(m(t-1) - m(t)),
    l(t) = alpha l(t-1) + sum exp(s_j - m(t)), o(t) = alpha o(t-1) + sum
    exp(s_j - m(t)) v_j.  A state whose max is still -inf contributes nothing
    (alpha = 1, p = 0).  Returns the list of states after each block and the
    final (O, lse).
    """
    n = s.shape[0]
    m = -np.inf
    ell = 0.0
    o = np.zeros(vals.shape[1], dtype=np.float64)
    states = []
    for t0 in range(0, n, block):
        sb = s[t0:t0 + block]
        m_new = max(m, float(sb.max()))
        if np.isinf(m_new):
            states.append((m, ell, o.copy()))
            continue
        alpha = np.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.where(np.isfinite(sb), np.exp(sb - m_new), 0.0)
        ell = alpha * ell + p.sum()
        o = _rescale(alpha, o) + p @ vals[t0:t0 + block]
        m = m_new
        states.append((m, ell, o.copy()))
    if ell == 0.0:
        return states, np.zeros_like(o), -np.inf
    return states, o / ell, m + np.log(ell)


def merge(state1, state2):
    """Combine two partial softmax states (m, l, o) over disjoint key sets."""
    m1, l1, o1 = state1
    m2, l2, o2 = state2
    m = max(m1, m2)
    if np.isinf(m):
        return m, 0.0, np.zeros_like(o1)
    a1 = np.exp(m1 - m) if np.isfinite(m1) else 0.0
    a2 = np.exp(m2 - m) if np.isfinite(m2) else 0.0
    return m, a1 * l1 + a2 * l2, a1 * o1 + a2 * o2


def partial_state(s, vals):
    """Unnormalised softmax state (m, l, o) of one key block, from scratch."""
    m = float(s.max())
    if np.isinf(m):
        return m, 0.0, np.zeros(vals.shape[1])
    p = np.where(np.isfinite(s), np.exp(s - m), 0.0)
    return m, float(p.sum()), p @ vals
