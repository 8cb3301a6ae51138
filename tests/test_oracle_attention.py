"""Pins for the three-pass float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a worked
example printed on "Learn: The Memory Wall & FlashAttention" (section 10,
practice problem 2), closed forms, invariants stated on the pages, a
high-precision decimal sum, and library routines (scipy, torch's CPU SDPA).
"""
import decimal
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "online_softmax_worked_example.json")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- worked example

def test_worked_example_printed_numbers():
    g = json.load(open(GOLDEN))
    s = np.array(g["scores"])
    vals = np.array(g["values"])[:, None]
    states, out, lse = oa.online_row(s, vals, g["block"])
    tol = 0.5 * 10.0 ** -g["printed_decimals"]
    m1, l1, o1 = states[0]
    m2, l2, o2 = states[1]
    assert m1 == g["after_block_1"]["m"] and m2 == g["after_block_2"]["m"]
    assert abs(l1 - g["after_block_1"]["ell"]) <= tol
    assert abs(o1[0] - g["after_block_1"]["o"]) <= tol
    assert abs(math.exp(m1 - m2) - g["after_block_2"]["alpha"]) <= tol
    assert abs(l2 - g["after_block_2"]["ell"]) <= tol
    assert abs(o2[0] - g["after_block_2"]["o"]) <= tol
    assert abs(out[0] - g["output"]) <= 5e-4           # printed with 3 decimals

    # The three-pass oracle on the same problem: d = 1, q = 1, k_j = s_j, scale 1.
    q = np.ones((1, 1))
    k = s[:, None]
    O3, L3 = oa.three_pass_rows(q, k, vals, 1.0, False, [0])
    assert abs(O3[0, 0] - g["output"]) <= 5e-4
    assert abs(L3[0] - (g["after_block_2"]["m"] + math.log(g["after_block_2"]["ell"]))) <= 1e-4
    # Direct weights exp(s_j - max) as printed.
    P = oa.probabilities(q, k, 1.0, False)[0]
    assert np.allclose(P * g["after_block_2"]["ell"], g["direct_weights"], atol=tol)


# ------------------------------------------------- three-pass == online == merge

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (7, 3), (33, 8), (64, 5)])
def test_three_pass_equals_online_and_merge(N, d, causal):
    q, k, v = (_rand((N, d), 10 + i) for i in range(3))
    scale = 0.7
    O3, L3 = oa.three_pass_rows(q, k, v, scale, causal, np.arange(N))
    for i in range(N):
        s = scale * (k @ q[i])
        if causal:
            s = np.where(np.arange(N) <= i, s, -np.inf)
        for block in sorted({1, 2, 3, N}):
            _, o, lse = oa.online_row(s, v, block)
            np.testing.assert_allclose(o, O3[i], rtol=1e-12, atol=1e-13)
            assert abs(lse - L3[i]) <= 1e-12 * max(1.0, abs(L3[i]))
        # Blockwise merge of two partial states, every split point.
        for cut in range(1, N):
            st = oa.merge(oa.partial_state(s[:cut], v[:cut]), oa.partial_state(s[cut:], v[cut:]))
            m, ell, acc = st
            np.testing.assert_allclose(acc / ell, O3[i], rtol=1e-12, atol=1e-13)
            assert abs(m + math.log(ell) - L3[i]) <= 1e-12 * max(1.0, abs(L3[i]))


def test_dropping_alpha_breaks_the_recurrence(monkeypatch):
    """Exercise 2 on the FA2 page: deferring alpha on the accumulator is wrong
    whenever the running max changes; the pin above must catch it."""
    s = np.array([1.0, 3.0, 4.0, 2.0])
    vals = np.array([[1.0], [2.0], [3.0], [4.0]])
    _, good, _ = oa.online_row(s, vals, 2)
    monkeypatch.setattr(oa, "_rescale", lambda alpha, acc: acc)
    _, bad, _ = oa.online_row(s, vals, 2)
    assert abs(bad[0] - good[0]) > 1e-2          # the max moved from 3 to 4
    # When the max never moves after the first block the mutation is harmless.
    s2 = np.array([4.0, 3.0, 1.0, 2.0])
    _, bad2, _ = oa.online_row(s2, vals, 2)
    O3, _ = oa.three_pass_rows(np.ones((1, 1)), s2[:, None], vals, 1.0, False, [0])
    assert abs(bad2[0] - O3[0, 0]) < 1e-12


# ----------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    N, d = 19, 6
    q = _rand((N, d), 1)
    k = np.repeat(_rand((1, d), 2), N, axis=0)
    v = _rand((N, d), 3)
    scale = 0.3
    O, L = oa.three_pass_rows(q, k, v, scale, causal, np.arange(N))
    for i in range(N):
        n_vis = i + 1 if causal else N
        np.testing.assert_allclose(O[i], v[:n_vis].mean(axis=0), rtol=1e-12, atol=1e-14)
        assert abs(L[i] - (scale * q[i] @ k[0] + math.log(n_vis))) <= 1e-12


def test_probability_rows_sum_to_one_and_match_lse():
    N, d = 40, 8
    q, k, v = (_rand((N, d), 20 + i) for i in range(3))
    for causal in (False, True):
        P = oa.probabilities(q, k, 0.5, causal)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
        _, L = oa.three_pass_rows(q, k, v, 0.5, causal, np.arange(N))
        S = 0.5 * q @ k.T
        if causal:
            S = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None], S, -np.inf)
        np.testing.assert_allclose(np.exp(S - L[:, None]), P, atol=1e-13)


def test_causal_row_zero_and_last_row():
    N, d = 50, 16
    q, k, v = (_rand((N, d), 30 + i) for i in range(3))
    scale = 1 / 4
    Oc, Lc = oa.three_pass_rows(q, k, v, scale, True, np.arange(N))
    On, Ln = oa.three_pass_rows(q, k, v, scale, False, np.arange(N))
    assert np.array_equal(Oc[0], v[0])
    assert abs(Lc[0] - scale * q[0] @ k[0]) <= 1e-15
    np.testing.assert_allclose(Oc[-1], On[-1], rtol=1e-13, atol=1e-15)
    assert abs(Lc[-1] - Ln[-1]) <= 1e-13


def test_lse_matches_decimal_sum():
    """lse_i = log sum_j exp(s_ij), against a 50-digit decimal evaluation."""
    N, d = 12, 4
    q, k, v = (_rand((N, d), 40 + i) for i in range(3))
    scale = 0.9
    _, L = oa.three_pass_rows(q, k, v, scale, False, np.arange(N))
    decimal.getcontext().prec = 50
    for i in range(N):
        tot = sum(decimal.Decimal(float(scale * (q[i] @ k[j]))).exp() for j in range(N))
        assert abs(float(tot.ln()) - L[i]) <= 1e-14


def test_one_huge_score_and_constant_values():
    N, d = 30, 8
    q, k, v = (_rand((N, d), 50 + i) for i in range(3))
    S = q @ k.T
    top2 = np.sort(S, axis=1)[:, -2:]
    scale = 60.0 / (top2[:, 1] - top2[:, 0]).min()     # every row's winner leads by >= 60
    O, _ = oa.three_pass_rows(q, k, v, scale, False, np.arange(N))
    np.testing.assert_allclose(O, v[S.argmax(axis=1)], atol=1e-20 + 1e-24 * scale)
    const = np.full((N, d), 2.5)
    for causal in (False, True):
        Oc, _ = oa.three_pass_rows(q, k, const, 0.4, causal, np.arange(N))
        np.testing.assert_allclose(Oc, 2.5, rtol=1e-14)


def test_key_value_permutation_invariance():
    N, d = 37, 8
    q, k, v = (_rand((N, d), 60 + i) for i in range(3))
    perm = np.random.default_rng(0).permutation(N)
    O1, L1 = oa.three_pass_rows(q, k, v, 0.35, False, np.arange(N))
    O2, L2 = oa.three_pass_rows(q, k[perm], v[perm], 0.35, False, np.arange(N))
    np.testing.assert_allclose(O1, O2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L1, L2, rtol=1e-14)


# ----------------------------------------------------------- library routines

@pytest.mark.parametrize("causal", [False, True])
def test_matches_scipy_softmax_and_logsumexp(causal):
    N, d = 70, 16
    q, k, v = (_rand((N, d), 70 + i) for i in range(3))
    scale = 1 / 4
    S = scale * q @ k.T
    if causal:
        S = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None], S, -np.inf)
    O, L = oa.three_pass_rows(q, k, v, scale, causal, np.arange(N))
    np.testing.assert_allclose(O, scipy.special.softmax(S, axis=1) @ v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L, scipy.special.logsumexp(S, axis=1), rtol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    B, H, N, d = 2, 3, 45, 8
    q, k, v = (_rand((B, H, N, d), 80 + i) for i in range(3))
    O, _ = oa.attention(q, k, v, d ** -0.5, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-11, atol=1e-13)


def test_row_subset_equals_full():
    B, H, N, d = 1, 2, 300, 8
    q, k, v = (_rand((B, H, N, d), 90 + i) for i in range(3))
    rows = [0, 5, 127, 128, 299]
    O, L = oa.attention(q, k, v, 0.3, True)
    Os, Ls = oa.attention(q, k, v, 0.3, True, rows=rows)
    np.testing.assert_array_equal(Os, O[:, :, rows])
    np.testing.assert_array_equal(Ls, L[:, :, rows])


# ----------------------------------------------- grouped-query heads, window

def test_gqa_equals_mha_with_repeated_kv_heads():
    B, H, H_kv, N, d = 2, 6, 2, 40, 8
    q = _rand((B, H, N, d), 100)
    k, v = _rand((B, H_kv, N, d), 101), _rand((B, H_kv, N, d), 102)
    for causal in (False, True):
        O, L = oa.attention(q, k, v, 0.4, causal)
        kr, vr = np.repeat(k, H // H_kv, axis=1), np.repeat(v, H // H_kv, axis=1)
        O2, L2 = oa.attention(q, kr, vr, 0.4, causal)
        np.testing.assert_array_equal(O, O2)
        np.testing.assert_array_equal(L, L2)
    with pytest.raises(ValueError):
        oa.attention(q, _rand((B, 4, N, d), 1), _rand((B, 4, N, d), 2), 0.4, False)


def test_window_special_cases():
    N, d = 50, 8
    q, k, v = (_rand((1, 1, N, d), 110 + i) for i in range(3))
    Oc, Lc = oa.attention(q, k, v, 0.3, True)
    Ow, Lw = oa.attention(q, k, v, 0.3, True, window=N)
    np.testing.assert_array_equal(Ow, Oc)
    np.testing.assert_array_equal(Lw, Lc)
    O1, L1 = oa.attention(q, k, v, 0.3, True, window=1)       # only the diagonal key
    np.testing.assert_array_equal(O1[0, 0], v[0, 0])
    np.testing.assert_allclose(L1[0, 0], 0.3 * np.einsum("nd,nd->n", q[0, 0], k[0, 0]), rtol=1e-14)


def test_window_row_equals_non_causal_on_its_key_slice():
    """Row i with window w sees exactly keys max(0, i-w+1)..i: the non-causal
    oracle on that slice must give the same row."""
    N, d, w = 70, 8, 13
    q, k, v = (_rand((N, d), 120 + i) for i in range(3))
    Ow, Lw = oa.three_pass_rows(q, k, v, 0.5, True, np.arange(N), window=w)
    for i in range(N):
        lo = max(0, i - w + 1)
        O1, L1 = oa.three_pass_rows(q[i:i + 1], k[lo:i + 1], v[lo:i + 1], 0.5, False, [0])
        np.testing.assert_allclose(Ow[i], O1[0], rtol=1e-12, atol=1e-14)
        assert abs(Lw[i] - L1[0]) <= 1e-12 * max(1.0, abs(L1[0]))
