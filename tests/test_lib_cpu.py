"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and its host-side logic (argument validation, schedule arithmetic,
status strings) behaves as include/attn.h states.  No kernel is launched."""
import ctypes
import os
import re

import pytest

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return ga.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        s = ga.status_str(code)
        assert s and s != "unknown status"
    assert ga.status_str(123) == "unknown status"


def test_schedule_arithmetic(L):
    assert ga.num_units(2, 16, 8192) == 2 * 16 * 32
    assert ga.num_units(1, 2, 256) == 2
    assert ga.num_units(1, 1, 257) == 2
    assert ga.num_units(1, 1, 1) == 1
    assert ga.grid_size(2, 16, 8192, 152) == 152
    assert ga.grid_size(1, 2, 256, 152) == 2
    assert ga.num_units(0, 1, 1) == 0


A = ctypes.c_void_p(0x10000)       # 16-byte aligned dummy addresses: never dereferenced,
M = ctypes.c_void_p(0x10002)       # validation fails before any CUDA call


def _fwd(L, q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=128, d=128, scale=0.1, causal=0, dtype=0):
    return L.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, None)


def test_validation_codes(L):
    assert _fwd(L, q=None) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, B=0) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, N=-1) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, scale=float("nan")) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, scale=float("inf")) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, causal=2) == ga.ATTN_ERR_INVALID_ARG
    assert _fwd(L, d=96) == ga.ATTN_ERR_UNSUPPORTED
    assert _fwd(L, dtype=1) == ga.ATTN_ERR_UNSUPPORTED
    assert _fwd(L, k=M) == ga.ATTN_ERR_ALIGNMENT
    assert _fwd(L, o=M) == ga.ATTN_ERR_ALIGNMENT
    assert L.attn_fp8_prep(A, A, A, None, 1, 1, 128, 64, 0, None) == ga.ATTN_ERR_UNSUPPORTED
    assert L.attn_fp8_prep(A, A, A, None, 1, 1, 128, 128, 2, None) == ga.ATTN_ERR_INVALID_ARG
    assert L.attn_fp8_prep(M, A, A, None, 1, 1, 128, 128, 0, None) == ga.ATTN_ERR_ALIGNMENT
    assert L.attn_fwd_fp8(A, A, A, A, A, None, A, None, 1, 1, 128, 128, 0.1, 0,
                          None) == ga.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_debug(A, A, A, A, None, 1, 1, 128, 128, 0.1, 0, None, 1000, 0,
                            None) == ga.ATTN_ERR_INVALID_ARG


def test_every_finite_scale_is_accepted(L):
    """Negative and zero scales are valid (the header defines them); only
    non-finite ones are refused.  A misaligned O makes every call stop at the
    alignment check, which comes after the scale check, so nothing launches."""
    for scale in (-1.0, -0.125, 0.0, -0.0, 1e-30, 3.0):
        assert _fwd(L, o=M, scale=scale) == ga.ATTN_ERR_ALIGNMENT, scale
    for scale in (float("nan"), float("inf"), float("-inf")):
        assert _fwd(L, o=M, scale=scale) == ga.ATTN_ERR_INVALID_ARG, scale


def test_ex_validation_codes(L):
    ex = lambda H=4, H_kv=2, causal=1, window=0, d=128: L.attn_fwd_ex(
        A, A, A, A, None, 1, H, H_kv, 256, d, 0.1, causal, window, 0, None)
    assert ex(H_kv=3) == ga.ATTN_ERR_INVALID_ARG      # does not divide H
    assert ex(H_kv=0) == ga.ATTN_ERR_INVALID_ARG
    assert ex(window=-1) == ga.ATTN_ERR_INVALID_ARG
    assert ex(causal=0, window=64) == ga.ATTN_ERR_INVALID_ARG   # windows are causal
    assert ex(d=96) == ga.ATTN_ERR_UNSUPPORTED


def test_window_flops_convention():
    from exact_attention_forward_fwd_gb300 import inputs
    w = inputs.WORKLOADS["n8192_d128_gqa4_window4096"]
    pairs = sum(min(i + 1, 4096) for i in range(8192))
    assert w.flops == 4.0 * 2 * 16 * 128 * pairs
    q, k, v = inputs.make_qkv(1, 4, 16, 64, seed=1, H_kv=2)
    assert q.shape == (1, 4, 16, 64) and k.shape == v.shape == (1, 2, 16, 64)


def test_valid_args_without_gpu_report_no_device(L):
    """All checks pass, so the device query runs: with no GPU it reports a
    CUDA error (or 'unsupported' on a non-sm_103 device), never success."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(L) in (ga.ATTN_ERR_CUDA, ga.ATTN_ERR_UNSUPPORTED)


def test_product_path_has_no_cpu_fallback():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ga.attn_fwd(q, q, q)


def test_splitkv_workspace_and_default_splits(L):
    """Host arithmetic of the split-KV contract: workspace = partial O (f32) and
    partial lse (f32), each rounded up to 256 bytes; the default split count is
    1 when the plain schedule fills the SMs, else the smallest S (capped by the
    128-key blocks and by 64) minimising the finish time of the split units
    dealt in the kernel's order to the first free SM (blocks + 4 per unit, 1
    for an empty range) plus, for S > 1, S x B*H*N*d*8 / 8.8e6 for the merge."""
    def ws(B, H, N, d, S):
        rows = S * B * H * N
        up = lambda x: (x + 255) // 256 * 256
        return up(rows * d * 4) + up(rows * 4)
    for args in [(1, 2, 256, 64, 3), (2, 16, 8192, 128, 1), (1, 1, 1, 128, 64), (3, 5, 77, 64, 7)]:
        assert ga.splitkv_workspace_bytes(*args) == ws(*args), args
    for bad in [(0, 1, 1, 64, 1), (1, 1, 1, 96, 1), (1, 1, 1, 64, 0), (1, 1, 1, 64, 65)]:
        assert ga.splitkv_workspace_bytes(*bad) == 0, bad

    def finish(B, H, N, causal, S, sms):
        # plain list scheduling, SM loads kept as a sorted list
        npairs, nb_all = (N + 255) // 256, (N + 127) // 128
        pairs = range(npairs - 1, -1, -1) if causal else range(npairs)
        loads = [0] * sms
        for pr in pairs:
            nb = min(nb_all, 2 * pr + 2) if causal else nb_all
            for _ in range(B * H):
                for sp in range(S):
                    size = (sp + 1) * nb // S - sp * nb // S
                    loads[0] += size + 4 if size else 1
                    loads.sort()
        return max(loads)

    def expect(B, H, N, d, causal, sms):
        if B * H * ((N + 255) // 256) >= sms:
            return 1
        nb = (N + 127) // 128
        t = lambda S: finish(B, H, N, causal, S, sms) + (S * B * H * N * d * 8 / 8.8e6 if S > 1 else 0)
        return min(range(1, min(64, nb) + 1), key=lambda S: (t(S), S))
    cases = [(2, 16, 8192, 128, 0, 152), (1, 2, 8192, 128, 0, 152), (1, 2, 8192, 128, 1, 152),
             (1, 2, 256, 64, 0, 152), (1, 1, 32768, 64, 1, 152), (1, 1, 16384, 128, 0, 1000),
             (3, 1, 1000, 64, 1, 152), (1, 3, 77, 128, 0, 152), (1, 4, 4096, 128, 1, 132)]
    for c in cases:
        assert ga.splitkv_default_splits(*c) == expect(*c), c
    assert ga.splitkv_default_splits(2, 16, 8192, 128, 0, 152) == 1   # 1024 units already
    assert ga.splitkv_default_splits(1, 2, 8192, 128, 0, 152) == 2    # 64 units: 1 wave of 32-block units
    assert ga.splitkv_default_splits(1, 2, 8192, 128, 1, 152) == 4    # causal: shorter units pack tighter
    assert ga.splitkv_default_splits(1, 2, 256, 64, 0, 152) == 2      # capped by 2 key blocks
    assert ga.splitkv_default_splits(0, 1, 1, 128, 0, 152) == 0
    assert ga.splitkv_default_splits(1, 1, 1, 96, 0, 152) == 0        # head dim 64 or 128 only


def test_splitkv_validation_codes(L):
    """Argument errors are reported before any device query."""
    f = lambda S=2, ws=A, nbytes=1 << 30, d=128: L.attn_fwd_splitkv(
        A, A, A, A, None, 1, 2, 2, 256, d, 0.1, 0, 0, 0, S, ws, nbytes, None)
    assert f(S=0) == ga.ATTN_ERR_INVALID_ARG
    assert f(S=65) == ga.ATTN_ERR_INVALID_ARG
    assert f(ws=None) == ga.ATTN_ERR_INVALID_ARG
    assert f(nbytes=ga.splitkv_workspace_bytes(1, 2, 256, 128, 2) - 1) == ga.ATTN_ERR_INVALID_ARG
    assert f(ws=ctypes.c_void_p(A.value + 8)) == ga.ATTN_ERR_ALIGNMENT
    assert f(d=96) == ga.ATTN_ERR_UNSUPPORTED


def test_bwd_workspace_and_validation(L):
    Npad = lambda N: (N + 127) // 128 * 128
    up = lambda x: (x + 255) // 256 * 256
    for B, H, N, d in [(1, 2, 300, 64), (2, 16, 8192, 128), (1, 1, 1, 128)]:
        assert ga.bwd_workspace_bytes(B, H, N, d) == 2 * up(B * H * Npad(N) * 4)
    assert ga.bwd_workspace_bytes(1, 1, 1, 96) == 0
    f = lambda lse=A, ws=A, nbytes=1 << 30, d=128, H_kv=2, causal=0, window=0: L.attn_bwd(
        A, A, A, A, lse, A, A, A, A, 1, 2, H_kv, 256, d, 0.1, causal, window, ws, nbytes, None)
    assert f(lse=None) == ga.ATTN_ERR_INVALID_ARG
    assert f(ws=None) == ga.ATTN_ERR_INVALID_ARG
    assert f(nbytes=ga.bwd_workspace_bytes(1, 2, 256, 128) - 1) == ga.ATTN_ERR_INVALID_ARG
    assert f(H_kv=3) == ga.ATTN_ERR_INVALID_ARG
    assert f(window=5) == ga.ATTN_ERR_INVALID_ARG
    assert f(d=96) == ga.ATTN_ERR_UNSUPPORTED
    assert f(ws=ctypes.c_void_p(A.value + 8)) == ga.ATTN_ERR_ALIGNMENT
