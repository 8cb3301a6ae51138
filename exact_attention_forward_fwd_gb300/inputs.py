"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It holds random-number generation and the workload catalogue only:
none of the attention arithmetic lives here, so the CPU oracle and the CUDA
path stay independent of each other.

Recipe (every tensor is [B, H, N, d], row-major, d innermost):
  * Q, K, V: i.i.d. N(0, 1) float32 draws from a ``torch.Generator`` seeded with
    ``seed * 16 + {0, 1, 2}``, rounded to bfloat16 (round-to-nearest-even).
  * ``k_scale``: K multiplied by a power of two after rounding (exact in bf16);
    the 2048-token workload uses 8 to stress the running max.
  * ``outlier_frac``: for each of Q, K, V, ``round(frac * numel)`` positions are
    drawn without replacement (stream ``seed * 16 + {3, 4, 5}``) and replaced by
    ``sign * U(10, 30)`` with a fair sign, then rounded to bfloat16.
  * Per-head random signs for the incoherent-processing rotation: an [H, d]
    int8 tensor of +-1 from stream ``seed * 16 + 6``.  The rotation is a random
    draw of the method, so it is generated here and handed to both sides.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-forward workload: shape, mode and input recipe."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dtype: str = "bf16"          # "bf16" or "fp8" (E4M3 operands, bf16 output)
    seed: int = 1000
    k_scale: float = 1.0
    outlier_frac: float = 0.0
    H_kv: int = 0              # KV heads (0: same as H)
    window: int = 0            # causal sliding window in keys (0: none)

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved for causal (the usual attention-forward convention);
        with a sliding window, 4*d per visible (query, key) pair."""
        if self.window > 0:
            n, w = self.N, min(self.window, self.N)
            pairs = w * (w + 1) / 2 + (n - w) * w
            return 4.0 * self.B * self.H * self.d * pairs
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f


# The five workloads: the small parity case, the 2048-token case (causal,
# non-causal and the K*8 running-max stress), the 8192-token head-dim-128 case,
# the 32768-token causal head-dim-64 case and the FP8 case with outliers.
WORKLOADS = {
    "n256_d64": Workload("n256_d64", 1, 2, 256, 64, False, seed=1001),
    "n2048_d128": Workload("n2048_d128", 4, 16, 2048, 128, False, seed=1002),
    "n2048_d128_causal": Workload("n2048_d128_causal", 4, 16, 2048, 128, True, seed=1002),
    "n2048_d128_k8": Workload("n2048_d128_k8", 4, 16, 2048, 128, False, seed=1002, k_scale=8.0),
    "n2048_d128_k8_causal": Workload("n2048_d128_k8_causal", 4, 16, 2048, 128, True, seed=1002,
                                     k_scale=8.0),
    "n8192_d128": Workload("n8192_d128", 2, 16, 8192, 128, False, seed=1003),
    "n8192_d128_causal": Workload("n8192_d128_causal", 2, 16, 8192, 128, True, seed=1003),
    "n32768_d64_causal": Workload("n32768_d64_causal", 1, 8, 32768, 64, True, seed=1004),
    "fp8_n8192_d128": Workload("fp8_n8192_d128", 2, 16, 8192, 128, False, dtype="fp8",
                               seed=1005, outlier_frac=0.001),
    # Grouped-query heads (16 query heads share 4 KV heads) with a causal 4096-key
    # sliding window, the shape of the FA2/3 page's flash_attn_func example.
    "n8192_d128_gqa4_window4096": Workload("n8192_d128_gqa4_window4096", 2, 16, 8192, 128, True,
                                           seed=1006, H_kv=4, window=4096),
    # One sequence of two heads: 64 query-tile pairs, fewer than the SMs of the
    # device -- the shape split-KV (FlashDecoding-style key splitting) is for.
    "n8192_d128_b1h2": Workload("n8192_d128_b1h2", 1, 2, 8192, 128, False, seed=1007),
    "n8192_d128_b1h2_causal": Workload("n8192_d128_b1h2_causal", 1, 2, 8192, 128, True, seed=1007),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _inject_outliers(x: torch.Tensor, frac: float, seed: int) -> torch.Tensor:
    n = x.numel()
    count = int(round(frac * n))
    if count == 0:
        return x
    g = _gen(seed)
    pos = torch.randperm(n, generator=g)[:count]
    mag = 10.0 + 20.0 * torch.rand(count, generator=g, dtype=torch.float64)
    sign = torch.where(torch.rand(count, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    flat = x.reshape(-1).clone()
    flat[pos] = (sign * mag).to(torch.float32)
    return flat.reshape(x.shape)


def make_qkv(B: int, H: int, N: int, d: int, seed: int, k_scale: float = 1.0,
             outlier_frac: float = 0.0, H_kv: int = 0):
    """Return (q, k, v) as bfloat16 CPU tensors: q [B, H, N, d], k and v
    [B, H_kv, N, d] (H_kv = H when 0)."""
    shapes = [(B, H, N, d), (B, H_kv or H, N, d), (B, H_kv or H, N, d)]
    out = []
    for i in range(3):
        x = torch.randn(shapes[i], generator=_gen(seed * 16 + i), dtype=torch.float32)
        if outlier_frac:
            x = _inject_outliers(x, outlier_frac, seed * 16 + 3 + i)
        out.append(x.to(torch.bfloat16))
    q, k, v = out
    if k_scale != 1.0:
        assert math.log2(k_scale).is_integer(), "k_scale must be a power of two"
        k = (k.to(torch.float32) * k_scale).to(torch.bfloat16)
    return q, k, v


def make_signs(H: int, d: int, seed: int) -> torch.Tensor:
    """[H, d] int8 tensor of +-1: the random diagonal of the per-head rotation."""
    bits = torch.randint(0, 2, (H, d), generator=_gen(seed * 16 + 6), dtype=torch.int8)
    return (bits * 2 - 1).to(torch.int8)


def workload_inputs(w: Workload):
    """(q, k, v) for a catalogue workload, bfloat16 CPU tensors."""
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.k_scale, w.outlier_frac, w.H_kv)


def sample_rows(N: int, count: int, seed: int, tile: int = 128):
    """Row indices for sampled checks at full size.

    Always includes row 0, the last row and the rows on both sides of every
    ``tile`` boundary; the rest are drawn uniformly without replacement.
    """
    rows = {0, N - 1}
    for b in range(tile, N, tile):
        rows.update((b - 1, b))
    g = _gen(seed * 16 + 7)
    extra = torch.randperm(N, generator=g)[:count].tolist()
    rows.update(extra)
    return sorted(r for r in rows if 0 <= r < N)
