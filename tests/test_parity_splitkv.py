"""GPU parity of split-KV attention (attn_fwd_splitkv: key ranges as separate
work units, partial results merged with the (m, l, O) combination rule)
against the float64 oracle, plus its workspace contract."""
import numpy as np
import pytest
import torch

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import inputs
from oracle import attention as oa
from parity_util import assert_bf16_parity, f64, metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_fwd_gb300 import build
    build.build()
    assert ga.device_status(clear=True) == 0


def _run(q, k, v, causal, splits, window=0, rows=None, scale=None):
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o, lse = ga.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window,
                                 scale=scale, num_splits=splits)
    assert ga.device_status() == 0
    O_ref, L_ref = oa.attention(f64(q), f64(k), f64(v), scale, causal, rows=rows, window=window)
    o, lse = o.cpu(), lse.cpu()
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    return metrics(o, lse, O_ref, L_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(129, 2), (300, 3), (640, 2), (640, 5), (1000, 7)])
def test_small_shapes(N, splits, d, causal):
    q, k, v = inputs.make_qkv(1, 3, N, d, seed=N * 11 + d + splits + int(causal))
    # Causal rows near the start see a few keys: O of unit size (gate beyond its rounding).
    assert_bf16_parity(_run(q, k, v, causal, splits), f"N={N} S={splits} d={d} causal={causal}",
                       rounding_floor=causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [3, 5, 16, 64])
def test_more_splits_than_key_blocks(splits, causal):
    """N = 200 has two 128-key blocks: most ranges are empty and get weight 0."""
    q, k, v = inputs.make_qkv(2, 2, 200, 128, seed=splits + 100 * int(causal))
    assert_bf16_parity(_run(q, k, v, causal, splits), f"S={splits} causal={causal}",
                       rounding_floor=causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_one_split_equals_plain_path(d, causal):
    """One range: the merge multiplies by exp(0) = 1 and adds log(1) = 0, so O and
    lse are bit-identical to attn_fwd."""
    q, k, v = [t.cuda() for t in inputs.make_qkv(2, 4, 777, d, seed=31 + d)]
    o1, l1 = ga.attn_fwd(q, k, v, causal=causal)
    o2, l2 = ga.attn_fwd_splitkv(q, k, v, causal=causal, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("H_kv,window,splits", [(2, 300, 4), (1, 129, 3), (4, 5000, 6)])
def test_grouped_heads_and_window(H_kv, window, splits):
    q, _, _ = inputs.make_qkv(1, 4, 700, 128, seed=window)
    _, k, v = inputs.make_qkv(1, H_kv, 700, 128, seed=window + 1)
    H = q.shape[1]
    k_full = k.repeat_interleave(H // H_kv, dim=1)
    v_full = v.repeat_interleave(H // H_kv, dim=1)
    o, lse = ga.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True, window=window,
                                 num_splits=splits)
    assert ga.device_status() == 0
    O_ref, L_ref = oa.attention(f64(q), f64(k_full), f64(v_full), 128 ** -0.5, True, window=window)
    assert_bf16_parity(metrics(o.cpu(), lse.cpu(), O_ref, L_ref), f"H_kv={H_kv} w={window}",
                       rounding_floor=True)


@pytest.mark.parametrize("name", ["n8192_d128_b1h2", "n8192_d128_b1h2_causal"])
def test_workload_sampled_rows_default_splits(name):
    """The one-sequence, two-head 8192-token workload with the library's default
    split count (the benchmark's launch configuration)."""
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_inputs(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits = ga.splitkv_default_splits(w.B, w.H, w.N, w.d, w.causal, sms)
    assert splits > 1
    rows = inputs.sample_rows(w.N, 64, w.seed)
    m = _run(q, k, v, w.causal, splits, rows=rows, scale=w.scale)
    print(name, "splits", splits, m)
    assert_bf16_parity(m, name)


def test_long_sequence_splits():
    """One head of 2^17 + 77 tokens (causal, d = 64) in 8 key ranges: ranges of
    up to 16k keys per unit, the merge over them, and the ragged last tile, on
    rows sampled around every tile boundary.  (The library's default split
    count here is 1: the head alone has 513 units.)"""
    N = 131149
    q, k, v = inputs.make_qkv(1, 1, N, 64, seed=41)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ga.splitkv_default_splits(1, 1, N, 64, True, sms) == 1
    splits = 8
    rows = inputs.sample_rows(N, 32, 41)
    m = _run(q, k, v, True, splits, rows=rows)
    print("N=131149 splits", splits, m)
    assert_bf16_parity(m, f"N={N} splits={splits}")


def test_workspace_contents_do_not_matter_and_repeatable():
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 2, 1000, 128, seed=3)]
    need = ga.splitkv_workspace_bytes(1, 2, 1000, 128, 5)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN patterns
    o1, l1 = ga.attn_fwd_splitkv(q, k, v, causal=True, num_splits=5, workspace=ws)
    ws.zero_()
    o2, l2 = ga.attn_fwd_splitkv(q, k, v, causal=True, num_splits=5, workspace=ws)
    o3, l3 = ga.attn_fwd_splitkv(q, k, v, causal=True, num_splits=5, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o2, o3) and torch.equal(l2, l3)


def test_workspace_errors():
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 2, 300, 64, seed=4)]
    need = ga.splitkv_workspace_bytes(1, 2, 300, 64, 3)
    small = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ga.AttnError) as e:
        ga.attn_fwd_splitkv(q, k, v, num_splits=3, workspace=small)
    assert e.value.status == ga.ATTN_ERR_INVALID_ARG
    big = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ga.AttnError) as e:
        ga.attn_fwd_splitkv(q, k, v, num_splits=3, workspace=big[4:])
    assert e.value.status == ga.ATTN_ERR_ALIGNMENT
    for bad in (0, 65):
        with pytest.raises(ga.AttnError) as e:
            ga.attn_fwd_splitkv(q, k, v, num_splits=bad, workspace=big)
        assert e.value.status == ga.ATTN_ERR_INVALID_ARG
    assert ga.device_status() == 0
