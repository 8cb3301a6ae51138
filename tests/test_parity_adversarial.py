"""GPU parity on the adversarial cases the pages name for a softmax kernel --
"one huge score" and "all-equal scores" ("Learn: The Memory Wall &
FlashAttention", section 11, hands-on 1) -- and on every kind of scale the
boundary accepts, through the C ABI, element by element against the float64
oracle.

  * scale < 0 and scale = 0: the running max must be the max of the *scaled*
    scores (section 5.1), whatever the sign; scale = 0 gives uniform weights.
  * identical keys: O_i is the mean of the visible V rows, lse_i = s_i + ln n_i.
  * one dominant key per row (Q = K, large scale): O_i -> V_argmax; the
    dominant key of a causal row arrives in the row's last key block, so the
    running reference moves late and the retake / rescale path runs.
  * constant V: any weights that sum to one give O = that constant.
The same cases run through the FP8 path, which takes the block max first.
"""
import numpy as np
import pytest
import torch

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import inputs
from oracle import attention as oa
from parity_util import (assert_bf16_parity, assert_fp8_fidelity, assert_fp8_parity, f64,
                         metrics)
from retake_cases import retake_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_fwd_gb300 import build
    build.build()
    assert ga.device_status(clear=True) == 0


def _bf16(q, k, v, causal, scale, splits=0):
    if splits:
        o, lse = ga.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                                     num_splits=splits)
    else:
        o, lse = ga.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ga.device_status() == 0
    O_ref, L_ref = oa.attention(f64(q), f64(k), f64(v), scale, causal)
    return o.cpu(), lse.cpu(), metrics(o.cpu(), lse.cpu(), O_ref, L_ref)


def _fp8(q, k, v, causal, scale, seed):
    H = q.shape[1]
    signs = inputs.make_signs(H, 128, seed)
    o, lse = ga.attn_fwd_fp8_from_bf16(q.cuda(), k.cuda(), v.cuda(), signs.cuda(), causal=causal,
                                       scale=scale)
    torch.cuda.synchronize()
    assert ga.device_status() == 0
    O_ref, L_ref = oa.attention(f64(q), f64(k), f64(v), scale, causal)
    m = metrics(o.cpu(), lse.cpu(), O_ref, L_ref)
    from oracle import fp8 as ofp8
    prep = ofp8.prepare(f64(q), f64(k), f64(v), signs.numpy())
    Oq, Lq = oa.attention(ofp8.dequantize(prep["q8"], prep["q_scale"]),
                          ofp8.dequantize(prep["k8"], prep["k_scale"]),
                          ofp8.dequantize(prep["v8"], prep["v_scale"]), scale, causal)
    return o.cpu(), m, metrics(o.cpu(), lse.cpu(), Oq, Lq)


# ------------------------------------------------------------------ scales

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("which", ["-1/sqrt(d)", "-1", "0"])
def test_negative_and_zero_scale(which, causal, d):
    scale = {"-1/sqrt(d)": -d ** -0.5, "-1": -1.0, "0": 0.0}[which]
    q, k, v = inputs.make_qkv(2, 2, 300, d, seed=700 + d + int(causal))
    _, _, m = _bf16(q, k, v, causal, scale)
    print(f"scale={which} d={d} causal={causal}: {m}")
    # scale -1 gives nearly one-hot rows and scale 0 averages a few keys in the
    # first causal rows: outputs of unit size, gate beyond their bf16 rounding.
    assert_bf16_parity(m, f"scale={which} d={d} causal={causal}", rounding_floor=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale_is_positive_scale_on_negated_keys(d, causal):
    """scale * (q.k) = |scale| * (q.(-k)) exactly, and negating bf16 keys is
    exact: the kernel's two ways of computing it give identical bits."""
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 3, 555, d, seed=710 + d))
    s = d ** -0.5
    o1, l1 = ga.attn_fwd(q, k, v, causal=causal, scale=-s)
    o2, l2 = ga.attn_fwd(q, -k, v, causal=causal, scale=s)
    torch.cuda.synchronize()
    assert ga.device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_zero_scale_closed_form():
    """scale = 0: O_i = mean of the visible V rows, lse_i = ln(visible count)."""
    N, d = 300, 128
    q, k, v = inputs.make_qkv(1, 2, N, d, seed=720)
    for causal in (False, True):
        o, lse, _ = _bf16(q, k, v, causal, 0.0)
        vv = f64(v)
        n = np.arange(1, N + 1) if causal else np.full(N, N)
        mean = np.cumsum(vv, axis=2) / n[None, None, :, None] if causal else \
            np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
        assert np.abs(f64(o) - mean).max() <= 1e-2 + 2 ** -8 * np.abs(mean).max()
        np.testing.assert_allclose(f64(lse), np.broadcast_to(np.log(n), (1, 2, N)), atol=1e-5)


@pytest.mark.parametrize("splits", [3, 7])
def test_negative_and_zero_scale_splitkv(splits):
    q, k, v = inputs.make_qkv(1, 2, 1000, 128, seed=730 + splits)
    for scale in (-128 ** -0.5, 0.0):
        _, _, m = _bf16(q, k, v, True, scale, splits=splits)
        assert_bf16_parity(m, f"split-KV S={splits} scale={scale}", rounding_floor=True)


def test_negative_and_zero_scale_grouped_heads_window():
    q, _, _ = inputs.make_qkv(1, 4, 700, 128, seed=740)
    _, k, v = inputs.make_qkv(1, 2, 700, 128, seed=741)
    kf, vf = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    for scale in (-128 ** -0.5, 0.0):
        o, lse = ga.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True, window=200, scale=scale)
        torch.cuda.synchronize()
        assert ga.device_status() == 0
        O_ref, L_ref = oa.attention(f64(q), f64(kf), f64(vf), scale, True, window=200)
        assert_bf16_parity(metrics(o.cpu(), lse.cpu(), O_ref, L_ref), f"GQA window scale={scale}",
                           rounding_floor=True)


# ---------------------------------------------------------- degenerate rows

def _identical_keys(B, H, N, d, seed):
    q, k, v = inputs.make_qkv(B, H, N, d, seed=seed)
    k = k[:, :, :1, :].expand(B, H, N, d).contiguous()
    return q, k, v


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale_sign", [1, -1])
def test_identical_keys(d, causal, scale_sign):
    """All keys equal: every visible score of row i is the same s_i, so
    O_i = mean of the visible V rows and lse_i = s_i + ln n_i."""
    N = 300
    q, k, v = _identical_keys(2, 2, N, d, seed=750 + d)
    scale = scale_sign * d ** -0.5
    o, lse, m = _bf16(q, k, v, causal, scale)
    assert_bf16_parity(m, f"identical keys d={d} causal={causal} sign={scale_sign}",
                       rounding_floor=causal)
    vv, s = f64(v), scale * np.einsum("bhnd,bhd->bhn", f64(q), f64(k)[:, :, 0, :])
    n = np.arange(1, N + 1) if causal else np.full(N, N)
    mean = np.cumsum(vv, axis=2) / n[None, None, :, None] if causal else \
        np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
    assert np.abs(f64(o) - mean).max() <= 1e-2 + 2 ** -8 * np.abs(mean).max()
    assert np.abs(f64(lse) - (s + np.log(n))).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [1.0, 4.0])
def test_one_dominant_key(d, causal, scale):
    """K = Q: q_i . q_i (about d) exceeds every other score of row i by ~90 at
    d = 128, so at scale >= 1 row i is one-hot on key i and O_i = v_i."""
    N = 1000
    q, _, v = inputs.make_qkv(1, 2, N, d, seed=760 + d)
    k = q.clone()
    o, lse, m = _bf16(q, k, v, causal, scale)
    assert_bf16_parity(m, f"dominant key d={d} causal={causal} scale={scale}", rounding_floor=True)
    vv = f64(v)
    assert np.abs(f64(o) - vv).max() <= 2 ** -8 * np.abs(vv).max()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_retake_with_weighty_earlier_keys(d, causal):
    """A block whose sum of p fails the 2^32 bound moves the reference to its
    max and is taken again, and what O and the sums already hold is rescaled.
    At d = 64 the kernel weighs a block's last 32 keys first and issues their
    P.V before testing the rest, so in head 0 those keys' product is already
    in O when the block fails; unlike the one-dominant-key case, the rescaled
    keys here keep a share of the row's weight (about 18 %) far above the
    gates, so a product rescaled wrongly, or rescaled before it landed, shows.
    Head 1 fails on its last keys alone, head 2 only moves the reference
    lazily.  Q is e_0 for every row and K's first column carries the scores."""
    N, H = 512, 3
    q = torch.zeros(1, H, N, d, dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = torch.zeros(1, H, N, d, dtype=torch.bfloat16)
    for h in range(H):
        k[0, h, :, 0] = retake_scores(h, N)
    _, _, v = inputs.make_qkv(1, H, N, d, seed=950 + d)
    o, lse, m = _bf16(q, k, v, causal, 1.0)
    assert_bf16_parity(m, f"retake d={d} causal={causal}")
    if not causal:
        # Head 0, every row: the rescaled last keys of block 2 weigh about 18 %.
        w = torch.softmax(retake_scores(0, N).double(), 0)
        assert 0.15 < float(w[352:384].sum()) < 0.21


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(d, causal):
    """Every V row the same vector c: O = c for any weights that sum to one."""
    q, k, v = inputs.make_qkv(2, 2, 640, d, seed=770 + d)
    v = v[:, :, :1, :].expand_as(v).contiguous()
    o, _, m = _bf16(q, k, v, causal, d ** -0.5)
    assert_bf16_parity(m, f"constant V d={d} causal={causal}", rounding_floor=True)
    c = f64(v)
    assert np.abs(f64(o) - c).max() <= 2 ** -8 * np.abs(c).max()


# -------------------------------------------------------------------- FP8
# The RMSE gate against the unquantised oracle holds where O averages many V
# rows.  Where a row is (nearly) one-hot or V is constant, O is one dequantised
# V row, whose E4M3 rounding alone is ~3.6 % RMS (3 mantissa bits): there only
# the kernel's fidelity to its own quantised operands is gated.

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [-128 ** -0.5, 0.0])
def test_fp8_negative_and_zero_scale(scale, causal):
    q, k, v = inputs.make_qkv(2, 2, 300, 128, seed=780 + int(causal))
    _, m, mq = _fp8(q, k, v, causal, scale, seed=780)
    print(f"fp8 scale={scale} causal={causal}: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_parity(m, f"fp8 scale={scale}")
    assert_fp8_fidelity(mq, f"fp8 scale={scale}")


def test_fp8_negative_scale_with_outliers():
    q, k, v = inputs.make_qkv(2, 2, 1024, 128, seed=782, outlier_frac=0.001)
    _, m, mq = _fp8(q, k, v, False, -128 ** -0.5, seed=782)
    print(f"fp8 scale=-1/sqrt(d), outliers: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_parity(m, "fp8 negative scale, outliers")
    assert_fp8_fidelity(mq, "fp8 negative scale, outliers")


def test_fp8_scale_minus_one_fidelity():
    q, k, v = inputs.make_qkv(2, 2, 300, 128, seed=785)
    _, m, mq = _fp8(q, k, v, True, -1.0, seed=785)
    print(f"fp8 scale=-1: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_fidelity(mq, "fp8 scale=-1")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_identical_keys(causal):
    q, k, v = _identical_keys(2, 2, 300, 128, seed=790)
    _, m, mq = _fp8(q, k, v, causal, 128 ** -0.5, seed=790)
    print(f"fp8 identical keys causal={causal}: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_parity(m, "fp8 identical keys")
    assert_fp8_fidelity(mq, "fp8 identical keys")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_constant_v(causal):
    q, k, v = inputs.make_qkv(2, 2, 300, 128, seed=791)
    v = v[:, :, :1, :].expand_as(v).contiguous()
    _, m, mq = _fp8(q, k, v, causal, 128 ** -0.5, seed=791)
    print(f"fp8 constant V causal={causal}: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_fidelity(mq, "fp8 constant V")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_one_dominant_key(causal):
    q, _, v = inputs.make_qkv(1, 2, 1000, 128, seed=795)
    k = q.clone()
    _, m, mq = _fp8(q, k, v, causal, 1.0, seed=795)
    print(f"fp8 dominant key causal={causal}: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_fidelity(mq, "fp8 dominant key")
