"""attn_fwd_splitkv_static: split-KV on the library's static scratch array.

The entry point is for callers that cannot call cudaMalloc (a host program that
owns all device memory through its own pool, or a loop that must not take
cudaMalloc's device-wide synchronisation), so its scratch is a fixed 64 MiB
device array inside the library.

Collected last on purpose (file name), and independent of every other test: it
must pass alone and after the rest of the suite.  It checks that two calls in a
row give exactly what attn_fwd_splitkv gives with a caller workspace (the
second call sees the first call's leftovers in the shared array), that a call
allocates no device memory, and that an oversize request is refused."""
import pytest
import torch

import exact_attention_forward_fwd_gb300 as ga
from exact_attention_forward_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_fwd_gb300 import build
    build.build()
    assert ga.device_status(clear=True) == 0


@pytest.mark.parametrize("B,H,N,d,causal,splits", [(1, 2, 1000, 128, True, 5),
                                                   (2, 3, 777, 64, False, 3),
                                                   (1, 2, 8192, 128, False, 7)])
def test_two_calls_in_a_row_match_workspace_entry(B, H, N, d, causal, splits):
    q, k, v = [t.cuda() for t in inputs.make_qkv(B, H, N, d, seed=N + splits)]
    ref_o, ref_l = ga.attn_fwd_splitkv(q, k, v, causal=causal, num_splits=splits)
    o1, l1 = ga.attn_fwd_splitkv_static(q, k, v, causal=causal, num_splits=splits)
    o2, l2 = ga.attn_fwd_splitkv_static(q, k, v, causal=causal, num_splits=splits)
    torch.cuda.synchronize()
    assert ga.device_status() == 0
    for o, l in ((o1, l1), (o2, l2)):
        assert torch.equal(o, ref_o)
        assert torch.equal(l, ref_l)


def test_fewer_splits_after_more_ignores_stale_partials():
    """A call with many key ranges leaves partial results all over the shared
    array; a following call with fewer ranges, several of them empty (causal
    pairs near the start have fewer key blocks than ranges), must read only
    what it wrote itself: bit for bit what attn_fwd_splitkv gives with a fresh
    workspace."""
    # 16 ranges x 4096 rows x 129 floats = 34 MB of the 64 MiB array.
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 1, 4096, 128, seed=41)]
    ga.attn_fwd_splitkv_static(q, k, v, causal=True, num_splits=16)
    for splits in (5, 3):
        ref_o, ref_l = ga.attn_fwd_splitkv(q, k, v, causal=True, num_splits=splits)
        o, l = ga.attn_fwd_splitkv_static(q, k, v, causal=True, num_splits=splits)
        torch.cuda.synchronize()
        assert ga.device_status() == 0
        assert torch.equal(o, ref_o)
        assert torch.equal(l, ref_l)


def test_call_allocates_no_device_memory():
    q, k, v = [t.cuda() for t in inputs.make_qkv(1, 2, 2048, 128, seed=9)]
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 2048, dtype=torch.float32, device="cuda")
    ga.attn_fwd_splitkv_static(q, k, v, num_splits=4, out=o, lse=lse)   # first call: address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        ga.attn_fwd_splitkv_static(q, k, v, num_splits=4, out=o, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    # torch's own count is exact; the device-wide free memory can also move
    # with other users of the GPU, so it only bounds an allocation of the
    # scratch's size (64 MiB) from below.
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 >= free0 - (8 << 20)


def test_oversize_request_is_refused():
    # 2 x 32 x 8192 rows x 129 floats x 2 splits ~ 270 MB > 64 MiB
    q, k, v = [torch.empty(2, 16, 8192, 128, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    assert ga.splitkv_workspace_bytes(2, 16, 8192, 128, 2) > (64 << 20)
    with pytest.raises(ga.AttnError) as e:
        ga.attn_fwd_splitkv_static(q, k, v, num_splits=2)
    assert e.value.status == ga.ATTN_ERR_INVALID_ARG
    assert ga.device_status() == 0

