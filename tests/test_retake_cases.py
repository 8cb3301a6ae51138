"""CPU checks of the constructed retake rows (no GPU): each head's scores take
the path of the kernel's reference rule its parity test relies on."""
import numpy as np
import pytest

from retake_cases import LOG2E, SUM_LIMIT, reference_path, retake_scores


def test_head0_retakes_after_its_last_keys_passed():
    ev = reference_path(retake_scores(0).float().numpy())
    assert [e[:2] for e in ev] == [(2, "block")]
    assert 0.15 < ev[0][2] < 0.21          # the rescaled last keys keep ~18 %


def test_head1_fails_on_its_last_keys_alone():
    ev = reference_path(retake_scores(1).float().numpy())
    assert [e[:2] for e in ev] == [(2, "tail")]


def test_head2_moves_lazily_without_retake():
    assert reference_path(retake_scores(2).float().numpy()) == []


def test_whole_block_rule_retakes_heads_0_and_1():
    """The d = 128 kernel tests whole blocks only: both heads retake there."""
    for h in (0, 1):
        ev = reference_path(retake_scores(h).float().numpy(), tail_first=False)
        assert [e[:2] for e in ev] == [(2, "block")]


# ---------------------------------------------------------------------------
# The d = 64 kernel's softmax algorithm restated in numpy (its order, not its
# code): per 128-key block, the last 32 keys are weighed first against the
# running reference m (and the block retaken on them alone if their sum
# passes 2^32), their P rounded to bf16 enters O and l~ at once, then the
# other 96 keys; if the whole block's sum fails the bound, O, l~ and l are
# rescaled by alpha = 2^(m_old - m_new) -- the last keys' contribution with
# them -- and only the other 96 keys are taken again.  Against the float64
# oracle this pins that weighing part of a block at the old reference and
# rescaling it afterwards is exact up to the bf16 rounding of P.

def _bf16(x):
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def early_tail_row(s, v, tail_first=True):
    """One row: s natural-unit scores (scale folded in), v [N, d] values.
    Returns (O, lse).  tail_first=False is the d = 128 kernel's order: the
    whole block is weighed and tested at once (its "last keys" are none)."""
    x_all = np.asarray(s, dtype=np.float64) * LOG2E
    m, ell, ellt = -np.inf, 0.0, 0.0
    o = np.zeros(v.shape[1])
    for j in range(len(x_all) // 128):
        x, vb = x_all[128 * j:128 * j + 128], v[128 * j:128 * j + 128]
        if m == -np.inf:
            m = x.max()
        t0 = 96 if tail_first else 128
        p_tail = np.exp2(x[t0:] - m)
        if p_tail.sum() > SUM_LIMIT:
            alpha = np.exp2(m - max(m, x.max()))
            m = max(m, x.max())
            o, ellt, ell = o * alpha, ellt * alpha, ell * alpha
            p_tail = np.exp2(x[t0:] - m)
        pb = _bf16(p_tail)
        o, ellt = o + pb @ vb[t0:], ellt + pb.sum()
        sum_tail = p_tail.sum()
        p_main = np.exp2(x[:t0] - m)
        if sum_tail + p_main.sum() > SUM_LIMIT:
            alpha = np.exp2(m - max(m, x.max()))
            m = max(m, x.max())
            o, ellt, ell = o * alpha, ellt * alpha, ell * alpha
            sum_tail *= alpha
            p_main = np.exp2(x[:t0] - m)
        pb = _bf16(p_main)
        o, ellt = o + pb @ vb[:t0], ellt + pb.sum()
        ell += sum_tail + p_main.sum()
    return o / ellt, (m + np.log2(ell)) / LOG2E


def _oracle_row(s, v):
    from oracle import attention as oa
    N, d = v.shape
    q = np.zeros((1, 1, N, 1)); k = np.zeros((1, 1, N, 1))
    q[0, 0, :, 0] = 1.0
    k[0, 0, :, 0] = s
    O, L = oa.attention(q, k, v[None, None], 1.0, False, rows=[0])
    return O[0, 0, 0], L[0, 0, 0]


@pytest.mark.parametrize("tail_first", [True, False])
def test_early_tail_algorithm_matches_the_oracle_on_the_retake_rows(tail_first):
    rng = np.random.default_rng(5)
    v = _bf16(rng.standard_normal((512, 64)))
    for head in (0, 1, 2):
        s = retake_scores(head).double().numpy()
        o, lse = early_tail_row(s, v, tail_first)
        O_ref, L_ref = _oracle_row(s, v)
        assert np.abs(o - O_ref).max() < 1e-2      # bf16 P: ~2^-9 relative per weight
        assert abs(lse - L_ref) < 1e-6             # l is summed in full precision here


@pytest.mark.parametrize("tail_first", [True, False])
def test_early_tail_algorithm_matches_the_oracle_on_random_rows(tail_first):
    rng = np.random.default_rng(6)
    for spread in (1.0, 8.0, 40.0):
        s = _bf16(rng.standard_normal(1024) * spread)
        v = _bf16(rng.standard_normal((1024, 64)))
        o, lse = early_tail_row(s, v, tail_first)
        O_ref, L_ref = _oracle_row(s, v)
        assert np.abs(o - O_ref).max() < 1e-2
        assert abs(lse - L_ref) < 1e-6


def test_early_tail_algorithm_needs_the_tail_rescaled():
    """Planting the mistake the ordering guards against -- the last keys'
    contribution left at the old reference when the block is retaken -- moves
    O far beyond the gates on head 0's rows."""
    rng = np.random.default_rng(5)
    v = _bf16(rng.standard_normal((512, 64)))
    s = retake_scores(0).double().numpy()
    x_all = s * LOG2E
    # the correct algorithm, then the same with the tail's product not rescaled
    o_ok, _ = early_tail_row(s, v)
    m = x_all[:128].max()
    o, ellt = np.zeros(64), 0.0
    for j in range(4):
        x, vb = x_all[128 * j:128 * j + 128], v[128 * j:128 * j + 128]
        pt = _bf16(np.exp2(x[96:] - m))
        tail_o, tail_l = pt @ vb[96:], pt.sum()
        if np.exp2(x - m).sum() > SUM_LIMIT:
            alpha = np.exp2(m - x.max())
            m = x.max()
            o, ellt = o * alpha, ellt * alpha      # the tail's product is NOT scaled here
        pm = _bf16(np.exp2(x[:96] - m))
        o, ellt = o + tail_o + pm @ vb[:96], ellt + tail_l + pm.sum()
    O_ref, _ = _oracle_row(s, v)
    assert np.abs(o_ok - O_ref).max() < 1e-2
    assert np.abs(o / ellt - O_ref).max() > 0.1
