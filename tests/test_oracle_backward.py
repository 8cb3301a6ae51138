"""Pins of the float64 backward oracle (oracle/backward.py) against things
other than itself: central finite differences of the (separately pinned)
forward oracle, torch autograd through torch's own softmax and matmul in
float64, closed forms and invariants of the softmax Jacobian, and the page's
identity D_i = rowdot(dO_i, O_i)."""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import backward as ob


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss_grad_fd(q, k, v, dO, scale, causal, window, eps=1e-6):
    """Central differences of L = sum(O * dO) with O from the forward oracle."""
    def loss(q_, k_, v_):
        O, _ = oa.attention(q_, k_, v_, scale, causal, window=window)
        return float((O * dO).sum())
    grads = []
    for which in range(3):
        base = [q, k, v][which]
        g = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p = [x.copy() for x in (q, k, v)]
            args_m = [x.copy() for x in (q, k, v)]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal,window,H,H_kv", [(False, 0, 1, 1), (True, 0, 1, 1),
                                                  (True, 3, 2, 1), (False, 0, 2, 2)])
def test_matches_finite_differences_of_forward_oracle(causal, window, H, H_kv):
    N, d, scale = 6, 3, 0.7
    q = _rand((1, H, N, d), 1)
    k = _rand((1, H_kv, N, d), 2)
    v = _rand((1, H_kv, N, d), 3)
    dO = _rand((1, H, N, d), 4)
    fd = _loss_grad_fd(q, k, v, dO, scale, causal, window)
    an = ob.backward(q, k, v, dO, scale, causal, window)
    for name, a, f in zip(("dQ", "dK", "dV"), an, fd):
        np.testing.assert_allclose(a, f, rtol=1e-6, atol=1e-7, err_msg=name)


def test_dropping_D_fails_the_finite_difference_pin():
    """A plausible mistake (dS = P o dP, the -D term dropped) is caught."""
    N, d, scale = 6, 3, 0.7
    q, k, v, dO = (_rand((1, 1, N, d), s) for s in (5, 6, 7, 8))
    fd = _loss_grad_fd(q, k, v, dO, scale, False, 0)
    P = ob.softmax_weights(q[0, 0], k[0, 0], scale, False)
    dS_wrong = P * (dO[0, 0] @ v[0, 0].T)
    dQ_wrong = scale * dS_wrong @ k[0, 0]
    assert np.abs(dQ_wrong - fd[0][0, 0]).max() > 1e-3


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 17)])
def test_matches_torch_autograd_float64(causal, window):
    B, H, H_kv, N, d, scale = 2, 4, 2, 70, 16, 0.25
    q, k, v = _rand((B, H, N, d), 11), _rand((B, H_kv, N, d), 12), _rand((B, H_kv, N, d), 13)
    dO = _rand((B, H, N, d), 14)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(H // H_kv, dim=1)
    vv = tv.repeat_interleave(H // H_kv, dim=1)
    S = scale * tq @ kk.transpose(-1, -2)
    if causal:
        i = torch.arange(N)[:, None]
        j = torch.arange(N)[None, :]
        vis = j <= i
        if window:
            vis &= j > i - window
        S = S.masked_fill(~vis, float("-inf"))
    O = torch.softmax(S, dim=-1) @ vv
    O.backward(torch.tensor(dO))
    an = ob.backward(q, k, v, dO, scale, causal, window)
    for name, a, t in zip(("dQ", "dK", "dV"), an, (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(a, t.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_page_identity_D_equals_rowdot_dO_O(causal):
    N, d, scale = 50, 8, 0.3
    q, k, v, dO = (_rand((N, d), s) for s in (21, 22, 23, 24))
    P = ob.softmax_weights(q, k, scale, causal)
    D_def = (P * (dO @ v.T)).sum(axis=1)
    O, _ = oa.attention(q[None, None], k[None, None], v[None, None], scale, causal)
    np.testing.assert_allclose(ob.row_dot(dO, O[0, 0]), D_def, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_jacobian_rows_sum_to_zero_so_dK_sums_to_zero(causal):
    """sum_j dS_ij = 0 for every row, hence sum over keys of dK = 0."""
    N, d, scale = 40, 5, 0.5
    q, k, v, dO = (_rand((N, d), s) for s in (31, 32, 33, 34))
    _, dK, dV = ob.backward_head(q, k, v, dO, scale, causal)
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-12)
    # Rows of P sum to 1, so the column sums of dV add up to the sum of dO.
    np.testing.assert_allclose(dV.sum(axis=0), dO.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_identical_keys_give_zero_dQ_and_mean_dO_dV():
    """All keys equal: P is uniform 1/N, S does not depend on q along the key
    axis, so dQ = 0 and dV_j = mean_i dO_i for every key j."""
    N, d = 30, 6
    q, v, dO = (_rand((N, d), s) for s in (41, 42, 43))
    k = np.tile(_rand((1, d), 44), (N, 1))
    dQ, dK, dV = ob.backward_head(q, k, v, dO, 0.8, False)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-12)
    np.testing.assert_allclose(dV, np.tile(dO.mean(axis=0), (N, 1)), rtol=1e-12, atol=1e-12)


def test_causal_row_zero_has_zero_dQ_and_last_key_sees_only_last_row():
    N, d, scale = 12, 4, 0.9
    q, k, v, dO = (_rand((N, d), s) for s in (51, 52, 53, 54))
    dQ, dK, dV = ob.backward_head(q, k, v, dO, scale, True)
    np.testing.assert_allclose(dQ[0], 0.0, atol=1e-14)          # one visible key: P = 1
    P = ob.softmax_weights(q, k, scale, True)
    np.testing.assert_allclose(dV[-1], P[-1, -1] * dO[-1], rtol=1e-12)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 9)])
def test_sampled_outputs_equal_full_backward(causal, window):
    N, d, scale = 700, 8, 0.4
    q, k, v, dO = (_rand((N, d), s) for s in (61, 62, 63, 64))
    dQ, dK, dV = ob.backward_head(q, k, v, dO, scale, causal, window)
    rows = [0, 1, 127, 128, 511, 512, 699]
    keys = [0, 5, 300, 698, 699]
    sq, sk, sv = ob.backward_sampled(q, k, v, dO, scale, causal, rows, keys, window)
    np.testing.assert_allclose(sq, dQ[rows], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sk, dK[keys], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sv, dV[keys], rtol=1e-10, atol=1e-12)
