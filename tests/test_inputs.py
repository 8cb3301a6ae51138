"""The seeded input generators: determinism, shapes and the outlier recipe."""
import torch

from exact_attention_forward_fwd_gb300 import inputs


def test_deterministic_and_shaped():
    a = inputs.make_qkv(1, 2, 130, 64, seed=7)
    b = inputs.make_qkv(1, 2, 130, 64, seed=7)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 130, 64)
        assert torch.equal(x, y)
    c = inputs.make_qkv(1, 2, 130, 64, seed=8)
    assert not torch.equal(a[0], c[0])


def test_k_scale_is_exact_power_of_two():
    q, k, v = inputs.make_qkv(1, 1, 64, 64, seed=3)
    _, k8, _ = inputs.make_qkv(1, 1, 64, 64, seed=3, k_scale=8.0)
    assert torch.equal(k8.float(), k.float() * 8)


def test_outliers_count_and_range():
    q, _, _ = inputs.make_qkv(1, 2, 500, 64, seed=5, outlier_frac=0.001)
    big = q.float().abs() >= 9.9
    assert int(big.sum()) == round(0.001 * q.numel())
    assert float(q.float().abs().max()) <= 30.5


def test_signs_and_rows():
    s = inputs.make_signs(4, 128, seed=9)
    assert s.dtype == torch.int8 and set(s.unique().tolist()) == {-1, 1}
    rows = inputs.sample_rows(1000, 10, seed=1)
    assert rows[0] == 0 and rows[-1] == 999 and 127 in rows and 128 in rows
