"""GPU parity of the attention backward (attn_bwd through the binding) against
the float64 backward oracle.

Gates (the acceptance criteria fix none for the backward; derived from the
arithmetic): P and dS enter the tensor-core products rounded to bf16 (relative
error <= 2^-9 each), the products accumulate in f32 and the outputs are rounded
to bf16.  A CPU simulation of exactly those roundings on the 2048-token
workloads (including the K x 8 variant, whose dQ is ~30 in magnitude) gives a
relative RMS error <= 4.5e-3 and a maximum error <= 2^-8 * max|ref|; the gates
are twice those: relative RMS <= 1e-2 and max |err| <= 2^-6 * max|ref| per
tensor (dQ, dK, dV), with the reference scale floored at 1e-3 (see FLOOR)."""
import numpy as np
import pytest
import torch

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import inputs
from oracle import attention as oa
from oracle import backward as ob
from parity_util import f64

pytestmark = pytest.mark.gpu

REL_RMSE = 1e-2
MAX_REL = 2.0 ** -6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_fwd_gb300 import build
    build.build()
    assert ga.device_status(clear=True) == 0


def _make_dO(B, H, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)


def _gpu_bwd(q, k, v, dO, causal, window=0, scale=None):
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, dO))
    if k.shape[1] != q.shape[1] or window:
        o, lse = ga.attn_fwd_ex(qc, kc, vc, causal=causal, window=window, scale=scale)
    else:
        o, lse = ga.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = ga.attn_bwd(qc, kc, vc, o, lse, dc, causal=causal, window=window, scale=scale)
    assert ga.device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


# Floor of the reference scale: a gradient that cancels to exactly zero (one
# visible key, identical keys) is matched to f32 rounding of its terms, O(1e-7)
# for these inputs, not to a fraction of zero.
FLOOR = 1e-3


def _check(name, got, ref):
    g = got.float().numpy().astype(np.float64)
    err = np.abs(g - ref)
    scale_ref = max(np.abs(ref).max(), FLOOR)
    rel_rmse = np.sqrt((err ** 2).mean()) / max(np.sqrt((ref ** 2).mean()), FLOOR)
    assert np.isfinite(g).all(), f"{name}: non-finite output"
    assert rel_rmse <= REL_RMSE, f"{name}: rel_rmse {rel_rmse:.3e}"
    assert err.max() <= MAX_REL * scale_ref, f"{name}: max err {err.max():.3e} (max|ref| {scale_ref:.3e})"
    return rel_rmse, err.max()


def _full(q, k, v, dO, causal, window=0, scale=None):
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = _gpu_bwd(q, k, v, dO, causal, window, scale)
    rq, rk, rv = ob.backward(f64(q), f64(k), f64(v), f64(dO), scale, causal, window)
    return [_check(n, gt, rf) for n, gt, rf in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv))]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 255, 256, 300, 640])
def test_small_shapes(N, d, causal):
    q, k, v = inputs.make_qkv(1, 2, N, d, seed=N * 13 + d + int(causal))
    dO = _make_dO(1, 2, N, d, seed=N + 1)
    _full(q, k, v, dO, causal)


@pytest.mark.parametrize("H_kv,window", [(1, 0), (2, 0), (2, 200), (4, 129)])
def test_grouped_heads_and_window(H_kv, window):
    q, _, _ = inputs.make_qkv(1, 4, 500, 128, seed=H_kv * 7 + window)
    _, k, v = inputs.make_qkv(1, H_kv, 500, 128, seed=H_kv * 7 + window + 1)
    dO = _make_dO(1, 4, 500, 128, seed=window + 3)
    _full(q, k, v, dO, causal=window > 0 or H_kv == 2, window=window)


@pytest.mark.parametrize("name", ["n2048_d128", "n2048_d128_causal", "n2048_d128_k8",
                                  "n2048_d128_k8_causal", "n256_d64"])
def test_workload_distributions(name):
    """Two heads with the workload's input recipe (the oracle backward is
    O(N^2 d) per head in float64)."""
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_qkv(1, 2, w.N, w.d, w.seed, w.k_scale)
    dO = _make_dO(1, 2, w.N, w.d, seed=w.seed + 50)
    res = _full(q, k, v, dO, w.causal, scale=w.scale)
    print(name, res)


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_sampled(causal):
    """The 8192-token head-dim-128 workload at full size (B=2, H=16), in the
    benchmark's launch configuration; dQ rows and dK, dV key rows sampled on
    two heads (row 0, the last row, both sides of 128-boundaries, random)."""
    w = inputs.WORKLOADS["n8192_d128_causal" if causal else "n8192_d128"]
    q, k, v = inputs.workload_inputs(w)
    dO = _make_dO(w.B, w.H, w.N, w.d, seed=w.seed + 60)
    dq, dk, dv = _gpu_bwd(q, k, v, dO, causal, scale=w.scale)
    rows = inputs.sample_rows(w.N, 24, w.seed)[::4]
    for (b, h) in [(0, 0), (1, 15)]:
        rq, rk, rv = ob.backward_sampled(f64(q)[b, h], f64(k)[b, h], f64(v)[b, h], f64(dO)[b, h],
                                         w.scale, causal, rows, rows)
        _check(f"dQ[{b},{h}]", dq[b, h, rows], rq)
        _check(f"dK[{b},{h}]", dk[b, h, rows], rk)
        _check(f"dV[{b},{h}]", dv[b, h, rows], rv)


def test_deterministic():
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 3, 700, 128, seed=8)]
    dO = _make_dO(1, 3, 700, 128, seed=9).cuda()
    o, lse = ga.attn_fwd(q, k, v, causal=True)
    a = ga.attn_bwd(q, k, v, o, lse, dO, causal=True)
    b = ga.attn_bwd(q, k, v, o, lse, dO, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_errors():
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 2, 300, 64, seed=2)]
    o, lse = ga.attn_fwd(q, k, v)
    dO = torch.zeros_like(q)
    need = ga.bwd_workspace_bytes(1, 2, 300, 64)
    with pytest.raises(ga.AttnError) as e:
        ga.attn_bwd(q, k, v, o, lse, dO, workspace=torch.empty(need - 1, dtype=torch.uint8,
                                                                 device="cuda"))
    assert e.value.status == ga.ATTN_ERR_INVALID_ARG
    rc = ga.lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None,
                           dO.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, 2, 2, 300,
                           64, 0.125, 0, 0, q.data_ptr(), need, None)
    assert rc == ga.ATTN_ERR_INVALID_ARG   # lse is required
    assert ga.device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [-1.0, -0.125, 0.0])
def test_negative_and_zero_scale(scale, d, causal):
    """The score products negate K (Q in the key-major kernel) for a negative
    scale, and dQ, dK carry the signed scale; scale = 0 gives uniform P, and
    dQ = dK = 0."""
    q, k, v = inputs.make_qkv(1, 2, 300, d, seed=900 + d + int(causal))
    dO = _make_dO(1, 2, 300, d, seed=901)
    _full(q, k, v, dO, causal, scale=scale)
