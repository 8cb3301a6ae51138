// Split-KV merge: combines the partial results of the key ranges of every query
// row into the final O (bf16) and logsumexp.
//
// The partial result of range s is (O_s, L_s) with O_s = sum_{i in s} p_i v_i /
// sum_{i in s} p_i and L_s = log sum_{i in s} exp(score_i), so with
// M = max_s L_s and w_s = exp(L_s - M):
//   O = sum_s w_s O_s / sum_s w_s,   L = M + log sum_s w_s.
// This is the rule for combining two blocks' (m, l, O) states ("FlashAttention-3
// & GPU Kernel Optimization: Accelerating Transformer Attention", section
// "Online softmax tiling mathematics"), applied along the key axis as in the
// FlashDecoding scheme ("4.3 FlashAttention 2 & 3", section "Comparison,
// trade-offs, and when each wins", paragraph on decode), written with the
// per-range logsumexp in place of the (m, l) pair.  A range that saw
// no visible key has L_s = -inf and weight 0; a row with no visible key at all
// gets O = 0 and L = -inf.
#include <cuda_runtime.h>

#include <cstdint>

#include "launchers.h"

namespace gb300 {

namespace {

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per query row; lane l owns head-dim elements [V*l, V*l + V).
template <int D>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part,
                                                            uint16_t* __restrict__ o,
                                                            float* __restrict__ lse, int S,
                                                            long long rows) {
  constexpr int V = D / 32;   // 4 (D = 128) or 2 (D = 64)
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float NEG_INF = __int_as_float(0xff800000);
  float M = NEG_INF;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldg(lse_part + s * rows + row));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  float den = 0.0f;
  if (M != NEG_INF) {
    for (int s = 0; s < S; ++s) {
      const float ls = __ldg(lse_part + s * rows + row);
      if (ls == NEG_INF) continue;   // empty range: weight 0
      const float w = expf(ls - M);
      den += w;
      const float* src = o_part + (static_cast<long long>(s) * rows + row) * D + V * lane;
      if (V == 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
        acc[2] = fmaf(w, x.z, acc[2]);
        acc[3] = fmaf(w, x.w, acc[3]);
      } else {
        const float2 x = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  const float inv = den > 0.0f ? 1.0f / den : 0.0f;
  uint16_t* dst = o + row * D + V * lane;
  if (V == 4) {
    const uint2 pk = make_uint2(bf16x2_rn(acc[0] * inv, acc[1] * inv), bf16x2_rn(acc[2] * inv, acc[3] * inv));
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = bf16x2_rn(acc[0] * inv, acc[1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[row] = den > 0.0f ? M + logf(den) : NEG_INF;
}

}  // namespace

cudaError_t launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                 int splits, int BH, int N, int D, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  constexpr int kWarps = 8;
  const long long blocks = (rows + kWarps - 1) / kWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  auto* out = reinterpret_cast<uint16_t*>(o);
  if (D == 128)
    splitkv_merge_kernel<128><<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
        o_part, lse_part, out, lse, splits, rows);
  else
    splitkv_merge_kernel<64><<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
        o_part, lse_part, out, lse, splits, rows);
  return cudaGetLastError();
}

}  // namespace gb300
