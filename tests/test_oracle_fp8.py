"""Pins for the Hadamard, E4M3 and FP8-preparation parts of the oracle (CPU only)."""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import e4m3, fp8, hadamard


# --------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("n", [1, 2, 4, 64, 128])
def test_sylvester_is_orthonormal_with_pm_entries(n):
    H = hadamard.sylvester(n)
    np.testing.assert_allclose(H @ H.T, np.eye(n), atol=1e-14)
    np.testing.assert_allclose(np.abs(H) * np.sqrt(n), 1.0, atol=1e-15)
    # Library routine: scipy's Sylvester-ordered Hadamard matrix.
    np.testing.assert_allclose(H, scipy.linalg.hadamard(n) / np.sqrt(n), atol=1e-15)


def test_small_textbook_matrix():
    r = 1 / np.sqrt(2)
    np.testing.assert_allclose(hadamard.sylvester(2), [[r, r], [r, -r]], atol=1e-16)


@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_fwht_equals_sylvester_on_basis_vectors(n):
    np.testing.assert_allclose(hadamard.fwht(np.eye(n)), hadamard.sylvester(n), atol=1e-15)
    x = np.random.default_rng(n).standard_normal((5, n))
    np.testing.assert_allclose(hadamard.fwht(x), x @ hadamard.sylvester(n), atol=1e-13)


def test_rotation_preserves_scores():
    d = 128
    rng = np.random.default_rng(1)
    Q, K = rng.standard_normal((64, d)), rng.standard_normal((64, d))
    signs = rng.choice([-1.0, 1.0], size=d)
    M = hadamard.rotation(signs)
    np.testing.assert_allclose((Q @ M) @ (K @ M).T, Q @ K.T, rtol=1e-12, atol=1e-11)


# ------------------------------------------------------------------ E4M3

def test_e4m3_named_codes():
    assert e4m3.decode_code(0x7E) == 448.0
    assert np.isnan(e4m3.decode_code(0x7F)) and np.isnan(e4m3.decode_code(0xFF))
    assert e4m3.decode_code(0x38) == 1.0
    assert e4m3.decode_code(0x01) == 2.0 ** -9
    assert e4m3.decode_code(0x08) == 2.0 ** -6
    assert e4m3.decode_code(0x07) == 7 / 8 * 2.0 ** -6
    assert e4m3.decode_code(0xFE) == -448.0
    assert e4m3.decode_code(0x80) == 0.0 and np.signbit(e4m3.decode_code(0x80))


def test_e4m3_all_codes_roundtrip():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3.decode(codes)
    back = e4m3.encode(vals)
    finite = ~np.isnan(vals)
    np.testing.assert_array_equal(back[finite], codes[finite])
    assert set(back[~finite].tolist()) == {0x7F, 0xFF}


def test_e4m3_ties_to_even_saturation_and_underflow():
    enc = lambda x: int(e4m3.encode(np.array([x]))[0])
    assert enc(1.0625) == 0x38            # halfway 1.0 / 1.125 -> even mantissa (1.0)
    assert enc(1.1875) == 0x3A            # halfway 1.125 / 1.25 -> 1.25
    assert enc(1.07) == 0x39              # nearest
    assert enc(1000.0) == 0x7E and enc(-1e9) == 0xFE and enc(460.0) == 0x7E
    assert enc(2.0 ** -11) == 0x00
    assert enc(2.0 ** -10) == 0x00        # halfway 0 / 2^-9 -> even code 0
    assert enc(3 * 2.0 ** -11) == 0x01    # nearer 2^-9 than 0
    assert enc(3 * 2.0 ** -10) == 0x02    # halfway 2^-9 / 2^-8 -> even code 2
    assert enc(5 * 2.0 ** -10) == 0x02    # halfway 2^-8 / 3*2^-9 -> even code 2
    assert enc(-2.0 ** -12) == 0x80       # sign kept on underflow
    assert enc(15 / 16 * 2.0 ** -6) == 0x08   # subnormal/normal tie -> even (normal)


def test_e4m3_matches_torch_float8_over_all_bf16():
    """Library routine: torch's float8_e4m3fn conversion on every finite bf16
    value of magnitude <= 448 (where saturation plays no part)."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(x) & (x.abs() <= 448)
    x = x[keep]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = e4m3.encode(x.to(torch.float64).numpy())
    np.testing.assert_array_equal(mine, ref)


# ---------------------------------------------------------- FP8 preparation

def test_block_scales_and_zero_block():
    x = np.zeros((1, 1, 300, 8))
    x[0, 0, 5, 3] = -7.0
    x[0, 0, 200, 1] = 3.0
    s = fp8.block_scales(x)
    assert s.shape == (1, 1, 3)
    assert s[0, 0, 0] == 7.0 / 448 and s[0, 0, 1] == 3.0 / 448 and s[0, 0, 2] == 1.0


def test_quantize_hits_448_and_error_bound():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 2, 260, 64)) * 3
    s = fp8.block_scales(x)
    c = fp8.quantize(x, s)
    deq = fp8.dequantize(c, s)
    for b in range(2):
        for h in range(2):
            for j in range(3):
                blk = e4m3.decode(c[b, h, 128 * j:128 * (j + 1)])
                assert np.abs(blk).max() == 448.0
    # Half a unit in the last place of E4M3: 2^-4 relative for normals,
    # 2^-10 * s absolute in the subnormal range.
    s_rows = np.repeat(s, 128, axis=2)[:, :, :260, None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s_rows) * (1 + 1e-12)
    assert np.all(np.abs(deq - x) <= bound)


def test_prepare_scores_invariant_and_outlier_gain():
    """Rotation leaves Q K^T unchanged; with an outlier feature (as in the FA2/3
    page's example) the rotated FP8 scores are closer to the exact ones."""
    rng = np.random.default_rng(4)
    B, H, N, d = 1, 2, 128, 128
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    q[..., 7] *= 25.0
    k[..., 7] *= 25.0
    v = rng.standard_normal((B, H, N, d))
    signs = rng.choice([-1.0, 1.0], size=(H, d))
    prep = fp8.prepare(q, k, v, signs)
    exact = np.einsum("bhnd,bhmd->bhnm", q, k)
    np.testing.assert_allclose(np.einsum("bhnd,bhmd->bhnm", prep["q_rot"], prep["k_rot"]),
                               exact, rtol=1e-10, atol=1e-9)
    rot = np.einsum("bhnd,bhmd->bhnm", fp8.dequantize(prep["q8"], prep["q_scale"]),
                    fp8.dequantize(prep["k8"], prep["k_scale"]))
    sq, sk = fp8.block_scales(q), fp8.block_scales(k)
    plain = np.einsum("bhnd,bhmd->bhnm", fp8.dequantize(fp8.quantize(q, sq), sq),
                      fp8.dequantize(fp8.quantize(k, sk), sk))
    assert np.abs(rot - exact).mean() < 0.5 * np.abs(plain - exact).mean()
