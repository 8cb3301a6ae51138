"""Failure detection without a GPU fault: a pipeline wait that runs out.

attn_fwd_debug makes the load warp stop after a few K/V tiles, so the MMA and
softmax waits on tiles that never arrive run out after a short limit.  The
kernel must then record ATTN_ERR_TIMEOUT in the caller's status word, free its
tensor memory and return; the context stays usable, which the follow-up
normal call checks against the oracle.  Nothing here traps, faults or hangs:
every wait in the kernel is bounded by a time limit.
"""
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


def test_debug_entry_without_fault_injection_matches_attn_fwd():
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 4, 640, 128, seed=21))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1 = ga.attn_fwd_debug(q, k, v, status, timeout_ns=1_000_000_000, skip_loads=0, causal=True)
    o2, l2 = ga.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert int(status.item()) == ga.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("skip", [1, 3, 10])
def test_missing_tiles_time_out_and_context_survives(skip):
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 8, 2048, 128, seed=22))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ga.attn_fwd_debug(q, k, v, status, timeout_ns=20_000_000, skip_loads=skip, causal=False)
    torch.cuda.synchronize()
    assert int(status.item()) == ga.ATTN_ERR_TIMEOUT
    # The library's own status word was not touched by the debug launch.
    assert ga.device_status(clear=True) == ga.ATTN_OK
    # A normal call afterwards runs correctly in the same context.
    qs, ks, vs = inputs.make_qkv(1, 2, 300, 64, seed=23)
    o, lse = ga.attn_fwd(qs.cuda(), ks.cuda(), vs.cuda(), causal=True)
    O, L = oa.attention(f64(qs), f64(ks), f64(vs), 64 ** -0.5, True)
    assert_bf16_parity(metrics(o.cpu(), lse.cpu(), O, L), "after timeout", rounding_floor=True)
