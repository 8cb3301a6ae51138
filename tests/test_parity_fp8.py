"""GPU parity of the FP8 path: the E4M3 preparation kernel against the
oracle's rotation / block scaling / E4M3 encoder, and the FP8 attention
forward against the float64 oracle run on the unquantised inputs."""
import numpy as np
import pytest
import torch

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import inputs
from oracle import attention as oa
from oracle import e4m3
from oracle import fp8 as ofp8
from parity_util import FP8_REL_RMSE, assert_fp8_fidelity, assert_fp8_parity, f64, metrics

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_fwd_gb300 import build
    build.build()


def _rows_view(codes, N, transpose):
    """GPU codes back in [B, H, N, d] order (and the padding of the transposed form)."""
    if not transpose:
        return codes, None
    return codes[..., :N].transpose(0, 1, 3, 2), codes[..., N:]


def test_e4m3_conversion_over_all_bf16_values():
    """With a 448 in every block the scale is exactly 1, so the kernel's codes
    must equal the oracle's RNE-satfinite encoding of every finite bf16 value
    of magnitude <= 448, bit for bit."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = bits.float()
    vals = vals[torch.isfinite(vals) & (vals.abs() <= 448)]
    per_block = 128 * 128 - 1
    nblk = -(-vals.numel() // per_block)
    x = torch.zeros(nblk, per_block)
    x.view(-1)[:vals.numel()] = vals
    x = torch.cat([torch.full((nblk, 1), 448.0), x], dim=1).reshape(1, 1, nblk * 128, 128)
    xb = x.to(torch.bfloat16)
    codes, sc = ga.fp8_prep(xb.cuda())
    assert torch.all(sc.cpu() == 1.0)
    ref = e4m3.encode(f64(xb))
    np.testing.assert_array_equal(codes.cpu().numpy(), ref)


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 300, 1024])
def test_prep_without_rotation_is_exact(N, transpose):
    """V path: codes decided in f32 (x / s, s = amax / 448) on both sides."""
    x, _, _ = inputs.make_qkv(2, 3, N, 128, seed=N + 3, outlier_frac=0.001)
    codes, sc = ga.fp8_prep(x.cuda(), None, transpose=transpose)
    codes, sc = codes.cpu().numpy(), sc.cpu().numpy()
    x32 = x.float().numpy()
    amax = ofp8.block_amax(x32.astype(np.float64)).astype(np.float32)
    s32 = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    np.testing.assert_array_equal(sc, s32)
    s_rows = np.repeat(s32, 128, axis=2)[:, :, :N, None]
    ref = e4m3.encode((x32 / s_rows).astype(np.float32).astype(np.float64))
    got, pad = _rows_view(codes, N, transpose)
    np.testing.assert_array_equal(got, ref)
    if pad is not None:
        assert not pad.any()


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 300, 1024])
def test_prep_with_rotation(N, transpose):
    """Q/K path: rotation computed in f32 by the kernel, in f64 by the oracle.
    Scales agree to f32 rounding; codes agree exactly except where the exact
    value lies within the f32 transform error bound of a rounding boundary,
    where the neighbouring code is also accepted (those cases are counted).
    The transposed output (any operand may ask for it) holds the same codes,
    and zeros in its padding."""
    B, H = 2, 3
    x, _, _ = inputs.make_qkv(B, H, N, 128, seed=N + 5, outlier_frac=0.001)
    signs = inputs.make_signs(H, 128, seed=N)
    codes, sc = ga.fp8_prep(x.cuda(), signs.cuda(), transpose=transpose)
    codes, pad = _rows_view(codes.cpu().numpy(), N, transpose)
    sc = sc.cpu().numpy().astype(np.float64)
    if pad is not None:
        assert not pad.any()
    xf = f64(x)
    xr = ofp8.rotate(xf, signs.numpy())
    s_ref = ofp8.block_scales(xr)
    # f32 error bound of the 7-stage butterfly plus the scaling products.
    row_l1 = np.abs(xf).sum(axis=-1, keepdims=True)
    e_x = 16 * U * row_l1 / np.sqrt(128) + 4 * U * np.abs(xr)
    amax_err = ofp8.block_amax(e_x)
    s_rel = amax_err / np.maximum(ofp8.block_amax(xr), 1e-300) + 4 * U
    np.testing.assert_allclose(sc, s_ref, rtol=float(s_rel.max()) + 1e-7)
    s_rows = np.repeat(s_ref, 128, axis=2)[:, :, :N, None]
    rel_rows = np.repeat(s_rel, 128, axis=2)[:, :, :N, None]
    y = xr / s_rows
    e_y = 2 * (e_x / s_rows + np.abs(y) * rel_rows)
    ref = e4m3.encode(y)
    diff = codes != ref
    if diff.any():
        gv, rv = e4m3.decode(codes[diff]), e4m3.decode(ref[diff])
        mid = 0.5 * (gv + rv)
        same_sign = np.signbit(gv) == np.signbit(rv)
        step = np.abs((codes[diff] & 0x7F).astype(int) - (ref[diff] & 0x7F).astype(int)) == 1
        near = np.abs(y[diff] - mid) <= e_y[diff]
        assert np.all(same_sign & step & near), "code mismatch outside the f32 error band"
    print(f"N={N}: {int(diff.sum())} boundary flips of {diff.size}")
    assert diff.sum() <= 1e-3 * diff.size


@pytest.mark.parametrize("transpose", [False, True])
def test_prep_tiny_and_zero_blocks(transpose):
    """Blocks whose scale s = amax / 448 is subnormal (amax ~ 1e-37, and bf16
    subnormal values), an all-zero block and a normal block: codes and scales
    equal the f32 arithmetic of the definition bit for bit (no reciprocal that
    overflows, no NaN codes)."""
    N = 4 * 128
    g = torch.Generator().manual_seed(77)
    x = torch.randn(1, 2, N, 128, generator=g)
    x[:, :, 128:256] *= 1e-37                       # s ~ 1e-37 / 448, subnormal
    x[:, :, 256:384] = 0.0                          # s = 1
    x[:, 1, 384:512] *= 1e-39                       # bf16 subnormal inputs
    x[:, :, 128:256:3] = 0.0                        # zeros inside a tiny block
    xb = x.to(torch.bfloat16)
    codes, sc = ga.fp8_prep(xb.cuda(), None, transpose=transpose)
    codes, sc = codes.cpu().numpy(), sc.cpu().numpy()
    x32 = xb.float().numpy()
    amax = ofp8.block_amax(x32.astype(np.float64)).astype(np.float32)
    s32 = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert (s32[:, :, 1] < np.float32(2.0 ** -126)).all()
    np.testing.assert_array_equal(sc, s32)
    s_rows = np.repeat(s32, 128, axis=2)[:, :, :N, None]
    with np.errstate(over="raise", invalid="raise"):
        y = (x32 / s_rows).astype(np.float32)
    ref = e4m3.encode(y.astype(np.float64))
    got, _ = _rows_view(codes, N, transpose)
    assert not np.isin(got, [0x7F, 0xFF]).any()
    np.testing.assert_array_equal(got, ref)


def test_prep_tiny_block_with_rotation():
    """The rotated path on a block of amax ~ 1e-37: finite codes, and the
    dequantised block within E4M3 resolution of the oracle's rotation."""
    N = 256
    g = torch.Generator().manual_seed(78)
    x = torch.randn(1, 2, N, 128, generator=g)
    x[:, :, 128:] *= 1e-37
    xb = x.to(torch.bfloat16)
    signs = inputs.make_signs(2, 128, seed=78)
    codes, sc = ga.fp8_prep(xb.cuda(), signs.cuda())
    codes, sc = codes.cpu().numpy(), sc.cpu().numpy().astype(np.float64)
    assert np.isfinite(sc).all() and (sc > 0).all()
    assert not np.isin(codes, [0x7F, 0xFF]).any()
    xr = ofp8.rotate(f64(xb), signs.numpy())
    deq = ofp8.dequantize(codes, sc)
    amax = np.repeat(ofp8.block_amax(xr), 128, axis=2)[:, :, :N, None]
    assert (np.abs(deq - xr) <= 2.0 ** -4 * amax).all()


def test_fp8_attention_on_the_oracles_operands():
    """The second FP8 check, kernel error alone: the attention kernel runs on
    the oracle's own E4M3 codes and block scales (uploaded; V only re-laid out
    as [d, Npad]), and is compared with the oracle on the same dequantised
    operands.  Prep rounding flips cannot enter: both sides read identical
    operands, so what remains is P's E4M3 rounding, f32 accumulation and the
    bf16 output."""
    B, H, N = 2, 2, 1000
    q, k, v = inputs.make_qkv(B, H, N, 128, seed=811, outlier_frac=0.001)
    signs = inputs.make_signs(H, 128, 811)
    prep = ofp8.prepare(f64(q), f64(k), f64(v), signs.numpy())
    nblk = (N + 127) // 128
    v8t = np.zeros((B, H, 128, nblk * 128), dtype=np.uint8)
    v8t[..., :N] = prep["v8"].transpose(0, 1, 3, 2)
    up = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()
    for causal in (False, True):
        o, lse = ga.attn_fwd_fp8(up(prep["q8"], torch.uint8), up(prep["k8"], torch.uint8),
                                 up(v8t, torch.uint8), up(prep["q_scale"], torch.float32),
                                 up(prep["k_scale"], torch.float32),
                                 up(prep["v_scale"], torch.float32), causal=causal)
        torch.cuda.synchronize()
        assert ga.device_status() == 0
        Oq, Lq = oa.attention(ofp8.dequantize(prep["q8"], prep["q_scale"]),
                              ofp8.dequantize(prep["k8"], prep["k_scale"]),
                              ofp8.dequantize(prep["v8"], prep["v_scale"]), 128 ** -0.5, causal)
        mq = metrics(o.cpu(), lse.cpu(), Oq, Lq)
        print(f"kernel alone, causal={causal}: {mq}")
        assert_fp8_fidelity(mq, f"oracle operands causal={causal}")


def _fp8_run(w_or_shape, rows=None):
    if isinstance(w_or_shape, inputs.Workload):
        w = w_or_shape
        q, k, v = inputs.workload_inputs(w)
        H, causal, scale, seed = w.H, w.causal, w.scale, w.seed
    else:
        B, H, N, causal, seed = w_or_shape
        q, k, v = inputs.make_qkv(B, H, N, 128, seed=seed, outlier_frac=0.001)
        scale = 128 ** -0.5
    signs = inputs.make_signs(H, 128, seed)
    o, lse = ga.attn_fwd_fp8_from_bf16(q.cuda(), k.cuda(), v.cuda(), signs.cuda(),
                                       causal=causal, scale=scale)
    assert ga.device_status() == 0
    O_ref, L_ref = oa.attention(f64(q), f64(k), f64(v), scale, causal, rows=rows)
    o, lse = o.cpu(), lse.cpu()
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    m = metrics(o, lse, O_ref, L_ref)
    # Diagnostic: against the oracle on the oracle's own quantised operands.
    prep = ofp8.prepare(f64(q), f64(k), f64(v), signs.numpy())
    Oq, Lq = oa.attention(ofp8.dequantize(prep["q8"], prep["q_scale"]),
                          ofp8.dequantize(prep["k8"], prep["k_scale"]),
                          ofp8.dequantize(prep["v8"], prep["v_scale"]), scale, causal, rows=rows)
    mq = metrics(o, lse, Oq, Lq)
    return m, mq


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 300, 1024])
def test_fp8_attention_small(N, causal):
    m, mq = _fp8_run((2, 2, N, causal, 40 + N))
    print(f"N={N} causal={causal}: vs exact {m}; vs quantised operands {mq}")
    assert_fp8_parity(m, f"N={N}")
    assert_fp8_fidelity(mq, f"N={N}")


def test_fp8_attention_workload_sampled_rows():
    w = inputs.WORKLOADS["fp8_n8192_d128"]
    rows = inputs.sample_rows(w.N, 64, w.seed)
    m, mq = _fp8_run(w, rows=rows)
    print(f"fp8 workload ({len(rows)} rows): vs exact {m}; vs quantised operands {mq}")
    assert_fp8_parity(m, w.name)
    assert_fp8_fidelity(mq, w.name)


def test_fp8_attention_long_sequence_sampled_rows():
    """FP8 on 2^16 + 5 tokens (prep and attention; ragged last block of the
    block scales and of V's transposed padding), rows sampled around every
    tile boundary.  The kernel's own error is gated against the oracle run on
    the same E4M3 operands (the second FP8 check), and the error against the
    exact result by its relative size.  The absolute RMSE gate of the FP8
    workload is not applied: on this input the E4M3 operands themselves (the
    method, with its 0.1 % outliers) put the exact result 0.029 away, which the
    kernel-only check separates out."""
    N = 65541
    rows = inputs.sample_rows(N, 32, 5)
    m, mq = _fp8_run((1, 1, N, False, 5), rows=rows)
    print(f"fp8 N={N} ({len(rows)} rows): vs exact {m}; vs quantised operands {mq}")
    assert m["finite"], "non-finite output"
    assert m["rel_rmse"] <= FP8_REL_RMSE, f"relative rmse {m['rel_rmse']:.3e}"
    assert_fp8_fidelity(mq, f"N={N}")


def test_fp8_writes_stay_inside_outputs():
    """The FP8 kernel's O (tensor stores, clipped at N) inside a larger buffer
    filled with a sentinel: nothing outside it changes, and the result equals
    the plain call's."""
    B, H, N, d, pad = 2, 2, 300, 128, 4096
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, N, d, seed=33))
    signs = inputs.make_signs(H, d, 33).cuda()
    q8, sq = ga.fp8_prep(q, signs)
    k8, sk = ga.fp8_prep(k, signs)
    v8, sv = ga.fp8_prep(v, None, transpose=True)
    n = B * H * N * d
    obuf = torch.full((n + 2 * pad,), 0x7E55, dtype=torch.int16, device="cuda")
    o = obuf[pad:pad + n].view(torch.bfloat16).view(B, H, N, d)
    ga.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=True, out=o)
    o_ref, _ = ga.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    torch.cuda.synchronize()
    assert ga.device_status() == 0
    assert torch.equal(o, o_ref)
    assert bool((obuf[:pad] == 0x7E55).all()) and bool((obuf[pad + n:] == 0x7E55).all())
